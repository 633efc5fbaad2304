#!/usr/bin/env python
"""Throughput of the GB300 dense GEMM with fused epilogue.

Headline workload (one "step" = one call of the whole hot path: host dispatch,
tile scheduler, TMA producer, tcgen05 MMA, fused epilogue and store):
    fp16 GEMM M = N = K = 4096, C = 1.5*A*B + 0.5*C, fp16 output, fp32
    accumulation, A, B ~ N(0,1)/sqrt(K), C ~ N(0,1) (seeded, synthetic).
Metric: TFLOP/s (2*M*N*K per step) and % of the GB300 dense tensor peak.

Timing: W untimed warm-up steps, then exactly K back-to-back steps between a
device synchronisation on both sides, bracketed by one pair of CUDA events on
the launch stream (``value`` = K steps of work over that time).  Three input
sets (288 MiB, more than the 129 MB L2) are used in rotation, so a step does
not find its operands in L2.  A separate pass of 30 calls, each between its
own events, gives the per-call median and bootstrap CI.

The library runs on one GPU: the path needs no exchange between GPUs (output
tiles are independent), so a multi-GPU job would be independent replicas, and
the pair kernel's TMA multicast is meant for single-GPU processes.  The bench
therefore refuses --gpus other than 1 and any torchrun launch with more than
one rank.

Besides the headline, the line carries one cell per workload configuration
(each timed as its own sequence of calls: median and bootstrap 95% CI of the
per-call TFLOP/s, inputs rotated through more than L2), the fused-vs-unfused
bias+GELU comparison, the cheap-baseline gate, the quantized decode cells, and
a short summary at its end.  Per-call samples of every cell go to a JSON file
beside the line (``--samples``).

``--impl reference`` times the float64 CPU oracle on the host cores on a
bounded row sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

REPO = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, REPO)

METRIC = "GEMM TFLOP/s at 4096³ (bf16/fp16, fp8) and % of GB300 dense tensor peak"
NOMINAL_PEAK_TFLOPS = {"f16": 2250.0, "bf16": 2250.0, "e4m3": 4500.0}
FALLBACK_BF16_TFLOPS = 1900.0
WORKLOAD = "fp16 GEMM M=N=K=4096, C=1.5*A*B+0.5*C, fp16 out, fp32 accumulation"
L2_BYTES = 129 * 10 ** 6  # GB300 L2 (the device property is used when a GPU is present)


def _args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--size", type=int, default=4096)
    ap.add_argument("--no-cells", action="store_true", help="skip the per-configuration cells")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle sample budget")
    ap.add_argument("--samples", default=None,
                    help="file for the per-call samples of every cell (default: bench_samples.json at the "
                         "repository root)")
    ap.add_argument("--profile", default=None, metavar="CASE",
                    help="run only CASE's workload --warmup + --steps times, untimed, for a profiler: "
                         + ", ".join(sorted(PROFILE_CASES)))
    ap.add_argument("--q4-decode", type=int, default=0, metavar="M",
                    help="only the quantized decode cell with M rows of x (for profiling); prints its JSON")
    ap.add_argument("--q4-reps", type=int, default=50, help="timed calls of the --q4-decode cell")
    ap.add_argument("--q4-kernel", choices=("auto", "ffma", "mma"), default="auto",
                    help="decode kernel of the --q4-decode cell")
    return ap.parse_args(argv)


# Workloads --profile runs (the cells' problems), by name.
PROFILE_CASES = {
    "headline": lambda wl: wl.fp16_alpha_beta(4096),
    "gelu_M512": lambda wl: wl.bf16_bias_gelu(512), "gelu_M2048": lambda wl: wl.bf16_bias_gelu(2048),
    "gelu_M8192": lambda wl: wl.bf16_bias_gelu(8192),
    "none_M2048": lambda wl: wl.bf16_bias_gelu(2048, epilogue=wl.EPI_NONE),
    "fp8_4096": lambda wl: wl.fp8_e4m3(4096), "fp8_8192": lambda wl: wl.fp8_e4m3(8192),
    "bf16_8192": lambda wl: wl.bf16_nn_large(8192), "fp32_4096_NN": lambda wl: wl.fp32_layout("NN", 4096),
    "mxfp8_4096": None, "mxfp4_4096": None, "q4_prefill_8192": None,
}


def run_profile(a):
    """--profile CASE: the case's calls back to back, nothing timed (for ncu)."""
    import torch
    import workloads as wl
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import dense_gemm_epilogues_tcgen05_gb300 as g
    stream = torch.cuda.current_stream()
    calls = a.warmup + a.steps
    if a.profile == "q4_prefill_8192":
        q4_prefill_cell(g, stream, 8192, steps=max(1, calls - 3))
        info = g.gemm_last_launch()
    elif a.profile.startswith("mx"):
        elem = wl.MX_E4M3 if a.profile.startswith("mxfp8") else wl.MX_E2M1
        mx_cell(g, stream, elem, 4096, steps=max(1, calls // 2), warmup=calls - max(1, calls // 2))
        info = g.gemm_last_launch()
    else:
        p = PROFILE_CASES[a.profile](wl)
        sets = _make_sets(p, 2, dev)
        for i in range(calls):
            _call(g, p, sets[i % 2], stream)
        torch.cuda.synchronize()
        info = g.gemm_last_launch()
    st = g.gemm_device_status()
    print(json.dumps({"profile": a.profile, "calls": calls, "status": st, "launch": info}), flush=True)
    if st != 0:
        raise SystemExit(1)


def workload_config(n):
    """The headline workload's description, the same for both arms."""
    mib = 3 * 3 * n * n * 2 / 2 ** 20
    return {"workload": WORKLOAD, "M": n, "N": n, "K": n, "layout": "A row-major (K-major), B row-major",
            "l2": f"3 rotating input sets ({mib:.0f} MiB, more than the 129 MB L2)", "parallelism": "single process"}


def refuse_multi_gpu(a, env=None):
    """The reason this process must not run (more than one GPU asked for), or None."""
    env = os.environ if env is None else env
    world = int(env.get("WORLD_SIZE", "1") or "1")
    if a.gpus != 1 or world != 1:
        return (f"bench.py runs on one GPU (asked: --gpus {a.gpus}, WORLD_SIZE {world}); the GEMM has no "
                f"exchange between GPUs, so N GPUs would be N independent replicas, and its TMA multicast "
                f"kernels are for single-GPU processes only")
    return None


# ----------------------------------------------------------------- helpers --

def bootstrap_ci(samples, reps=10000, seed=0, q=(2.5, 97.5)):
    """Median and percentile-bootstrap CI of the median (fixed seed, 10^4 resamples)."""
    import numpy as np
    x = np.asarray(samples, dtype=np.float64)
    if x.size == 0:
        return float("nan"), [float("nan"), float("nan")]
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, x.size, size=(reps, x.size))
    meds = np.median(x[idx], axis=1)
    return float(np.median(x)), [float(np.percentile(meds, q[0])), float(np.percentile(meds, q[1]))]


def bimodality(samples, min_share=0.05, min_sep=4.0, min_rel=0.02):
    """Two-mode test of per-call samples (Rigel section 3: clock states split small sizes into two
    modes).  The best split of the sorted samples into a low and a high group (least pooled
    variance) counts as two modes when each group holds at least `min_share` of the samples and
    the gap between their means exceeds `min_sep` pooled standard deviations and `min_rel` of the
    median.  Returns {"bimodal", "modes", "share"}."""
    import numpy as np
    x = np.sort(np.asarray(samples, dtype=np.float64))
    n = x.size
    if n < 10:
        return {"bimodal": False, "modes": [float(np.median(x))] if n else [], "share": [1.0] if n else []}
    c1, c2 = np.cumsum(x), np.cumsum(x * x)
    best = None
    lo_n = max(1, int(math.ceil(min_share * n)))
    for k in range(lo_n, n - lo_n + 1):
        m1, m2 = c1[k - 1] / k, (c1[-1] - c1[k - 1]) / (n - k)
        v1 = c2[k - 1] / k - m1 * m1
        v2 = (c2[-1] - c2[k - 1]) / (n - k) - m2 * m2
        pooled = (k * max(v1, 0.0) + (n - k) * max(v2, 0.0)) / n
        if best is None or pooled < best[0]:
            best = (pooled, k, m1, m2)
    pooled, k, m1, m2 = best
    sd = math.sqrt(pooled)
    med = float(np.median(x))
    two = (m2 - m1) > min_sep * sd and (m2 - m1) > min_rel * abs(med)
    if not two:
        return {"bimodal": False, "modes": [med], "share": [1.0]}
    return {"bimodal": True, "modes": [round(float(m1), 2), round(float(m2), 2)],
            "share": [round(k / n, 3), round((n - k) / n, 3)]}


def measured_peaks():
    path = os.path.join(REPO, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": float(d["bf16_tflops"]), "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]),
                "hbm_gbs": float(d["hbm_gbs"]), "sm_max_mhz": float(d.get("sm_max_mhz", 2070.0)),
                "source": "measured"}
    except Exception:
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
                "sm_max_mhz": 2070.0, "source": "fallback"}


def recorded_traffic(kernel_tag):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; otherwise None."""
    import __graft_entry__
    fp = __graft_entry__.build_module().source_fingerprint()[:16]
    path = os.path.join(REPO, "profiles", "dram_traffic.tsv")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.rstrip("\n").split("\t")
            if len(parts) >= 3 and parts[0] == fp and parts[1] == kernel_tag:
                return float(parts[2])
    return None


def aggregate(local_seconds, flops_per_step, steps, dist=None, device="cpu"):
    """Whole-job throughput: every rank ran `steps` steps of `flops_per_step`;
    the job's time is the slowest rank's.  Returns (TFLOP/s, max seconds).
    (The GEMM itself runs on one GPU; this is the aggregation rule a replica
    job would follow, kept with its CPU test.)"""
    import torch
    world = 1
    t = float(local_seconds)
    if dist is not None and dist.is_initialized():
        world = dist.get_world_size()
        x = torch.tensor([t], dtype=torch.float64, device=device)
        dist.all_reduce(x, op=dist.ReduceOp.MAX)
        t = float(x.item())
    return flops_per_step * steps * world / t / 1e12, t


def provenance(problem=None):
    """Where a number came from (Rigel section 3): source fingerprint, commit when
    the tree has one, input recipe and its hash, device, driver, CUDA and
    library versions, host cores."""
    import __graft_entry__
    out = {"sources": __graft_entry__.build_module().source_fingerprint()[:16]}
    try:
        r = subprocess.run(["git", "-C", REPO, "rev-parse", "--short=12", "HEAD"], capture_output=True, text=True,
                           timeout=5)
        if r.returncode == 0 and r.stdout.strip():
            out["commit"] = r.stdout.strip()
    except Exception:
        pass
    if problem is not None:
        out["recipe"] = problem.recipe
        out["recipe_hash"] = problem.recipe_hash()
    try:
        import torch
        out["torch"] = torch.__version__
        out["cuda"] = torch.version.cuda
        if torch.cuda.is_available():
            out["device"] = torch.cuda.get_device_name(0)
    except Exception:
        pass
    try:
        r = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader"],
                           capture_output=True, text=True, timeout=10)
        if r.returncode == 0:
            out["driver"] = r.stdout.strip().splitlines()[0]
    except Exception:
        pass
    out["host"] = platform.machine()
    out["cores"] = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return out


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.tmp is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.tmp.flush()
        with open(self.tmp.name) as f:
            text = f.read()
        os.unlink(self.tmp.name)
        return self.parse(text)

    @staticmethod
    def parse(text):
        """Summary of nvidia-smi CSV rows (the FIELDS order, no header, no units)."""
        rows = [r.split(",") for r in text.strip().splitlines() if r.strip()]
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0])); smax.append(float(r[1])); power.append(float(r[2]))
                for nm, val in zip(names, r[4:8]):
                    if val.strip().lower() in ("active", "1"):
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [s for s, p in zip(sm, power) if p > 0.3 * max(power)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


# ------------------------------------------------------------------ our arm --

_WS = {}


def _workspace(g, device, nbytes=0):
    """The library's workspace (stream-K scratch, or the 3xTF32 split of fp32
    operands), allocated outside any timed region and reused."""
    import torch
    key = str(device)
    need = max(nbytes, g.gemm_workspace_size(1, 1, 1, g.BF16), 256)
    if key not in _WS or _WS[key].numel() < need:
        _WS.pop(key, None)
        _WS[key] = torch.empty(need, dtype=torch.uint8, device=device)
    return _WS[key]


def set_bytes(p):
    """Device bytes of one input set of problem p (A, B, C, bias)."""
    n = p.A.numel() * p.A.element_size() + p.B.numel() * p.B.element_size() + p.C.numel() * p.C.element_size()
    return n + (0 if p.bias is None else p.bias.numel() * 4)


def sets_beyond_l2(p, l2_bytes=L2_BYTES, factor=1.5, cap=160):
    """How many input sets of p to rotate so their total exceeds factor x L2 (at least 2)."""
    return max(2, min(cap, int(math.ceil(factor * l2_bytes / max(1, set_bytes(p))))))


def _make_sets(problem, n_sets, device):
    import torch
    A, B, C = problem.A.to(device), problem.B.to(device), problem.C.to(device)
    bias = None if problem.bias is None else problem.bias.to(device)
    sets = [(A, B, C, bias)]
    for _ in range(n_sets - 1):
        sets.append((torch.empty_like(A).copy_(A), torch.empty_like(B).copy_(B), torch.empty_like(C).copy_(C),
                     None if bias is None else torch.empty_like(bias).copy_(bias)))
    return sets


def _call(g, p, s, stream, baseline=None, mode="fused"):
    A, B, C, bias = s
    if baseline is not None:
        g.gemm_baseline(baseline, p.M, p.N, p.K, p.ab_dtype, A, p.a_stride_m, p.a_stride_k, B, p.b_stride_k,
                        p.b_stride_n, C, p.ldc, p.c_dtype, p.alpha, p.beta, bias, p.epilogue, stream=stream)
        return
    ws = _workspace(g, C.device, g.gemm_workspace_size(p.M, p.N, p.K, p.ab_dtype))
    epi = p.epilogue if mode == "fused" else g.EPI_NONE
    g.gemm(p.M, p.N, p.K, p.ab_dtype, A, p.a_stride_m, p.a_stride_k, B, p.b_stride_k, p.b_stride_n, C, p.ldc,
           p.c_dtype, p.alpha, p.beta, bias, epi, workspace=ws, workspace_bytes=ws.numel(), stream=stream)
    if mode == "decomposed":
        # the unfused path: the plain GEMM, then the separate bias+GELU pass over C
        g.gemm_bias_gelu(p.M, p.N, C, p.ldc, p.c_dtype, bias, stream=stream)


def time_steps(g, p, sets, steps, warmup, stream, sampler=None, baseline=None, mode="fused"):
    """Warm up, then time `steps` calls, each between its own pair of events;
    returns (per-step ms list, total ms)."""
    import torch
    for i in range(warmup):
        _call(g, p, sets[i % len(sets)], stream, baseline, mode)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        torch.cuda.synchronize()
        ev[0].record(stream)
        for i in range(steps):
            _call(g, p, sets[i % len(sets)], stream, baseline, mode)
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return per, ev[0].elapsed_time(ev[steps])


def time_region(g, p, sets, steps, warmup, stream, sampler=None, baseline=None, mode="fused"):
    """Warm up, then time `steps` back-to-back calls between ONE pair of events
    (device synchronisation on both sides); returns total ms.  Nothing is
    recorded between the calls, so consecutive launches overlap as they do in
    a stream of GEMMs: the next grid's prologue starts while the previous one
    drains (programmatic dependent launch).  An event recorded between two
    launches orders them fully and costs about 5 % at 4096^3 (cuBLAS alike)."""
    import torch
    for i in range(warmup):
        _call(g, p, sets[i % len(sets)], stream, baseline, mode)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(steps):
            _call(g, p, sets[i % len(sets)], stream, baseline, mode)
        e1.record(stream)
        torch.cuda.synchronize()
    return e0.elapsed_time(e1)


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


SAMPLES = {}


def cell(g, p, steps, warmup, stream, n_sets=None, baseline=None, mode="fused", name=None, l2=L2_BYTES):
    """Time problem p (inputs rotated through more than L2) twice: `steps` calls
    back to back between one event pair ("tflops": the rate in a stream of such
    calls) and `steps` calls each between its own events (the per-call median
    and bootstrap CI).  The per-call samples are kept under `name`."""
    import torch
    n_sets = sets_beyond_l2(p, l2) if n_sets is None else n_sets
    sets = _make_sets(p, n_sets, torch.device("cuda", torch.cuda.current_device()))
    total = time_region(g, p, sets, steps, warmup, stream, baseline=baseline, mode=mode)
    per, _ = time_steps(g, p, sets, steps, 1, stream, baseline=baseline, mode=mode)
    tf = [p.flops / (t * 1e-3) / 1e12 for t in per]
    med, ci = bootstrap_ci(tf)
    del sets
    torch.cuda.empty_cache()
    if name is not None:
        SAMPLES[name] = [round(x, 2) for x in tf]
    return {"tflops": round(p.flops * steps / (total * 1e-3) / 1e12, 1), "ms": round(total / steps, 4),
            "per_call": {"median": round(med, 1), "ci95": [round(ci[0], 1), round(ci[1], 1)]}, "n": steps}


def paired_pct(num, den):
    """Median over rounds of 100 * (num_r / den_r - 1): rates taken side by side in each round."""
    return statistics.median(100.0 * (a / b - 1.0) for a, b in zip(num, den))


def interleaved_modes(g, p, modes, calls, rounds, stream, l2=L2_BYTES, name=None):
    """Time problem p in each of `modes` ("fused": its epilogue; "none": the plain GEMM; "decomposed":
    the plain GEMM, then the separate bias+GELU pass) in `rounds` alternating rounds, each mode
    `calls` calls back to back between one event pair per round, on the same inputs (rotated
    through more than L2).  Per mode: the median rate over rounds, and the per-call median and
    bootstrap CI from one pass with events around every call."""
    import torch
    sets = _make_sets(p, sets_beyond_l2(p, l2), torch.device("cuda", torch.cuda.current_device()))
    rates = {m: [] for m in modes}
    for r in range(rounds):
        for m in (modes if r % 2 == 0 else modes[::-1]):
            total = time_region(g, p, sets, calls, 3, stream, mode="plain" if m == "none" else m)
            rates[m].append(p.flops * calls / (total * 1e-3) / 1e12)
    out = {}
    for m in modes:
        per, _ = time_steps(g, p, sets, 30, 1, stream, mode="plain" if m == "none" else m)
        tf = [p.flops / (t * 1e-3) / 1e12 for t in per]
        med, ci = bootstrap_ci(tf)
        if name is not None:
            SAMPLES[f"{name}_{m}"] = [round(x, 2) for x in tf]
        rate = statistics.median(rates[m])
        out[m] = {"tflops": round(rate, 1), "ms": round(p.flops / (rate * 1e12) * 1e3, 4),
                  "rounds": [round(x, 1) for x in rates[m]],
                  "per_call": {"median": round(med, 1), "ci95": [round(ci[0], 1), round(ci[1], 1)]},
                  "n": calls * rounds}
    del sets
    torch.cuda.empty_cache()
    return out


def describe_launch(info):
    """One line for the roofline's kernel field, from gemm_last_launch()."""
    if info.get("kind") == 2:
        shape = {4: "two-pair clusters (A shared by TMA multicast)", 2: "one-pair clusters"}.get(
            info["cluster_ctas"], f"{info['cluster_ctas']}-CTA clusters")
        order = ", C^T = B^T A^T" if info.get("transposed") else ""
        sk = f", stream-K over {info['stream_k_tiles']} of {info['tiles']} units" if info.get("stream_k_tiles") else ""
        return (f"gemm_tcgen05_pair_kernel 256x{info['bn']} tiles, {shape}, {info['grid_ctas']} CTAs"
                f"{order}{sk}")
    if info.get("kind") == 1:
        return f"gemm_tcgen05_kernel 128x{info['bn']} tiles, {info['grid_ctas']} CTAs"
    return f"path {info.get('path')}"


def host_link_gbs(nbytes_in, nbytes_out, reps=10):
    """Measured pinned-host <-> device copy bandwidth (GB/s) for copies of these sizes, each
    direction alone (the bound an end-to-end step cannot beat)."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    h_in = torch.empty(nbytes_in, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes_in, dtype=torch.uint8, device=dev)
    h_out = torch.empty(nbytes_out, dtype=torch.uint8).pin_memory()
    d_out = torch.empty(nbytes_out, dtype=torch.uint8, device=dev)
    res = {}
    for name, dst, src, nb in (("h2d", d_in, h_in, nbytes_in), ("d2h", h_out, d_out, nbytes_out)):
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        res[name] = nb * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9
    return res


def e2e_measure(g, p, steps, stream):
    """Same metric through the public call with host buffers: every step copies
    its inputs A, B, C from pinned host memory, runs the GEMM and copies C back,
    all inside the timed region.  Steps are pipelined the way a serving loop
    would run them: copy-in, GEMM and copy-out each have a stream, device
    buffers alternate between two sets, and events order each step's three
    parts, so step i+1's copy-in overlaps step i's GEMM and step i-1's
    copy-out (the host-device link is the bound either way)."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    hA, hB, hC = p.A.pin_memory(), p.B.pin_memory(), p.C.clone().pin_memory()
    d_sets = [(torch.empty_like(hA, device=dev), torch.empty_like(hB, device=dev), torch.empty_like(hC, device=dev))
              for _ in range(2)]
    h_out = [torch.empty_like(hC).pin_memory() for _ in range(2)]
    bias = None
    ws = _workspace(g, dev)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]
    for e in ev_free:
        e.record(s_out)

    def step(i):
        b = i & 1
        dA, dB, dC = d_sets[b]
        s_in.wait_event(ev_free[b])  # the set's previous GEMM and copy-out are done
        with torch.cuda.stream(s_in):
            dA.copy_(hA, non_blocking=True)
            dB.copy_(hB, non_blocking=True)
            dC.copy_(hC, non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        g.gemm(p.M, p.N, p.K, p.ab_dtype, dA, p.a_stride_m, p.a_stride_k, dB, p.b_stride_k, p.b_stride_n, dC,
               p.ldc, p.c_dtype, p.alpha, p.beta, bias, p.epilogue, workspace=ws, workspace_bytes=ws.numel(),
               stream=stream)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            h_out[b].copy_(dC, non_blocking=True)
        ev_free[b].record(s_out)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(steps):
        step(i)
    s_in.wait_stream(s_out)  # e1 after every step's copy-out
    e1.record(s_in)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    h2d = hA.numel() * hA.element_size() + hB.numel() * hB.element_size() + hC.numel() * hC.element_size()
    d2h = h_out[0].numel() * h_out[0].element_size()
    link = host_link_gbs(h2d, d2h)
    h2d_gbs = h2d / (ms * 1e-3) / 1e9
    return {"value": round(p.flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "pipelined": "copy-in / GEMM / copy-out streams, two device buffer sets",
            "host_link": {"h2d_gbs": round(h2d_gbs, 1), "h2d_peak_gbs": round(link["h2d"], 1),
                          "frac": round(h2d_gbs / link["h2d"], 3), "d2h_peak_gbs": round(link["d2h"], 1),
                          "peak_source": "pinned copies of the same sizes, each direction alone"}}


def cpu_baseline(p, seconds, single_sample=False):
    """The float64 oracle, as it stands, on a bounded row sample of the workload."""
    import numpy as np
    import oracle
    args = p.oracle_args()
    rows_done, t_total, r = 0, 0.0, 16
    rng = np.random.default_rng(5)
    while t_total < seconds and rows_done < p.M:
        rows = np.sort(rng.choice(p.M, size=min(r, p.M - rows_done), replace=False))
        t0 = time.perf_counter()
        oracle.gemm_reference(rows=rows, **args)
        t_total += time.perf_counter() - t0
        rows_done += len(rows)
        if single_sample:
            break
        r = min(r * 2, 1024)
    flops = 2.0 * rows_done * p.N * p.K
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(flops / t_total / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows_done} of {p.M} output rows of the {p.M}x{p.N}x{p.K} workload "
                      f"(full K and N per row), {t_total:.1f} s", "seconds": round(t_total, 2)}


def run_ours(a):
    import torch
    import workloads as wl
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import dense_gemm_epilogues_tcgen05_gb300 as g

    n = a.size
    p = wl.fp16_alpha_beta(n)
    stream = torch.cuda.current_stream()
    sets = _make_sets(p, 3, dev)
    sampler = ClockSampler(0)
    total = time_region(g, p, sets, a.steps, a.warmup, stream, sampler=sampler)
    st = g.gemm_device_status()
    if st != 0:
        raise RuntimeError(f"device status after timing: {g.gemm_status_string(st)}")
    value, total_s = aggregate(total * 1e-3, p.flops, a.steps)
    # the per-call distribution (Rigel section 3: median and bootstrap CI over >= 30 reps), from
    # a separate pass with an event pair around every call
    per, _ = time_steps(g, p, sets, 30, 3, stream)
    tf = [p.flops / (t * 1e-3) / 1e12 for t in per]
    med, ci = bootstrap_ci(tf)
    peaks = measured_peaks()
    avg_ms = total / a.steps  # the kernel's average launch duration over the timed region
    achieved = p.flops / (avg_ms * 1e-3) / 1e12
    launch = g.gemm_last_launch()  # what the timed calls enqueued (the same call every step)
    kernel = describe_launch(launch)
    traffic = recorded_traffic("tcgen05_f16_4096")
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": round(total_s * 1e3 / a.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic: seeded A,B ~ N(0,1)/sqrt(K) fp16, C ~ N(0,1) fp16",
        "config": workload_config(n),
        "pct_of_nominal_peak": round(100 * value / NOMINAL_PEAK_TFLOPS["f16"], 2),
        "per_call": {"median_tflops": round(med, 2), "ci95": [round(ci[0], 2), round(ci[1], 2)], "n": len(tf),
                     "timing": "an event pair around each call (orders the launches fully)"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": traffic,
                     "peak_source": f"{peaks['source']} bf16 burst (fp16 runs at the bf16 rate)",
                     "kernel": kernel},
        "clocks": {**sampler.summary(), "region_ms": round(total, 3)},
        "gpu_launches": a.steps,
        "launch": launch,
        "provenance": provenance(p),
    }
    SAMPLES["headline"] = [round(x, 2) for x in tf]
    out["e2e"] = e2e_measure(g, p, 30, stream)
    del sets
    torch.cuda.empty_cache()
    if not a.no_cells:
        # The timed region above lasts a few milliseconds, less than nvidia-smi's sampling
        # period; the cells keep the GPU busy for about ten seconds, so their samples show the
        # clocks and throttle reasons under sustained load.
        cells_sampler = ClockSampler(0)
        with cells_sampler:
            cells, summary = extra_cells(g, stream, peaks)
        out["cells"] = cells
        out["clocks_cells"] = cells_sampler.summary()
    else:
        summary = {}
    out["cpu_baseline"] = cpu_baseline(p, a.cpu_seconds)
    summary["headline_tflops"] = round(value, 1)
    summary["headline_frac"] = out["roofline"]["frac"]
    out["summary"] = summary
    path = a.samples if a.samples is not None else os.path.join(REPO, "bench_samples.json")
    if path:
        try:
            with open(path, "w") as f:
                json.dump({"unit": "TFLOP/s per call (GB/s for q4 cells)", "samples": SAMPLES}, f)
            out["samples_file"] = os.path.relpath(path, REPO)
        except OSError:
            pass
    print(json.dumps(out), flush=True)


def extra_cells(g, stream, peaks):
    """One cell per workload configuration (fp16 sweep and ragged shape, fp8 with fp16 twins,
    fp32 layouts, bf16 and block-scaled inputs), the fused-vs-unfused
    bias+GELU comparison, the cheap-baseline gate and the quantized decode cells.
    Returns (cells, summary); the summary repeats the per-dtype headline figures."""
    import torch
    import workloads as wl
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size or L2_BYTES
    cells, summary = {}, {}

    def run(name, p, steps=30, warmup=5, **kw):
        c = cell(g, p, steps, warmup, stream, name=name, l2=l2, **kw)
        cells[name] = c
        return c

    # fp32 256^3 (3xTF32 with the workspace), latency-bound
    run("fp32_256", wl.fp32_square(256), steps=100, warmup=10)
    # fp16 alpha/beta sweep with ragged 1000^3; small sizes keep per-call samples and the two-mode test
    for n, reps in ((512, 300), (1024, 300), (2048, 100), (1000, 100)):
        c = run(f"fp16_{n}", wl.fp16_alpha_beta(n), steps=reps, warmup=20)
        if n in (512, 1024):
            c.update(bimodality(SAMPLES[f"fp16_{n}"]))
    # fused bias+GELU against the plain GEMM and against GEMM + the separate bias+GELU pass,
    # the three timed in alternating rounds on the same inputs (a cost of a few percent is below the
    # drift between two cells timed one after the other)
    gelu_cost, fusion_gain = {}, {}
    for M, calls in ((512, 200), (2048, 100), (8192, 30)):
        c = interleaved_modes(g, wl.bf16_bias_gelu(M), ("fused", "none", "decomposed"), calls, 8, stream, l2,
                              name=f"gelu_M{M}")
        # each round's modes ran next to each other: the median of the per-round ratios is
        # robust to the clock drifting between rounds (seen at M = 8192 under the power cap)
        cost = round(paired_pct(c["none"]["rounds"], c["fused"]["rounds"]), 2)
        gain = round(paired_pct(c["fused"]["rounds"], c["decomposed"]["rounds"]), 2)
        cells[f"gelu_M{M}"] = dict(c, fused_cost_pct=cost, fusion_gain_pct=gain)
        gelu_cost[M], fusion_gain[M] = cost, gain
    # fp32 layouts (3xTF32) with ldc padding, and bf16 8192^3 NN
    for lay in ("NN", "NT", "TN", "TT"):
        run(f"fp32_4096_{lay}", wl.fp32_layout(lay, 4096), steps=20, warmup=3)
    cells["baseline_gate_fp16_4096"] = baseline_gate(g, stream, l2)
    for M in (1, 2, 8):
        cells[f"q4_decode_M{M}"] = q4_decode_cell(g, stream, M, compact=True)
    for M in (64, 4096):
        cells[f"q4_prefill_M{M}"] = q4_prefill_cell(g, stream, M)
    # block-scaled MXFP8 / MXFP4, against 2x (fp8) and the fp4 rate
    mx = {}
    for nm, elem in (("mxfp8", wl.MX_E4M3), ("mxfp4", wl.MX_E2M1)):
        c = mx_cell(g, stream, elem, 4096, name=f"{nm}_4096")
        c["frac_of_2x_bf16_peak"] = round(c["tflops"] / (2 * peaks["bf16_tflops"]), 4)
        cells[f"{nm}_4096"] = c
        mx[nm] = c["tflops"]
    # fp8 with its fp16 twins (bf16 output, and an fp32-output cell) and the large
    # bf16 cells last, so that the tail of the line carries them
    fp8 = {}
    for n in (2048, 4096, 8192):
        steps = 30 if n < 8192 else 10
        c8 = run(f"fp8_{n}", wl.fp8_e4m3(n), steps=steps, warmup=3)
        c16 = run(f"fp16_twin_{n}", wl.fp16_twin_of_fp8(n), steps=steps, warmup=3)
        c8["over_fp16"] = round(c8["tflops"] / c16["tflops"], 3)
        c8["frac_of_2x_bf16_peak"] = round(c8["tflops"] / (2 * peaks["bf16_tflops"]), 4)
        fp8[n] = c8
    run("fp8_4096_f32out", wl.fp8_e4m3(4096, c_dtype=wl.F32), steps=30, warmup=3)
    bf = run("bf16_4096_nn", wl.bf16_nn_large(4096), steps=30, warmup=3)
    b8 = run("bf16_8192_nn", wl.bf16_nn_large(8192), steps=10, warmup=3)
    summary.update({
        "fp16_4096_gate_cell": cells["baseline_gate_fp16_4096"]["tcgen05"]["tflops"],
        "bf16_4096": bf["tflops"], "bf16_8192": b8["tflops"],
        "bf16_8192_frac": round(b8["tflops"] / peaks["bf16_tflops"], 4),
        "fp8_2048": fp8[2048]["tflops"], "fp8_4096": fp8[4096]["tflops"], "fp8_8192": fp8[8192]["tflops"],
        "fp8_over_fp16": {n: fp8[n]["over_fp16"] for n in fp8},
        "fp8_4096_frac_of_2x_bf16": fp8[4096]["frac_of_2x_bf16_peak"],
        "gelu_fused_cost_pct": gelu_cost, "gelu_fusion_gain_pct": fusion_gain,
        "q4_decode_frac": {M: cells[f"q4_decode_M{M}"]["frac"] for M in (1, 2, 8)},
        "mxfp8_4096": mx["mxfp8"], "mxfp4_4096": mx["mxfp4"],
    })
    return cells, summary


def mx_cell(g, stream, elem, n, steps=30, warmup=3, name=None):
    """Block-scaled product (gemm_mx) n^3, bf16 output: A, B ~ N(0,1) quantised to MX
    (OCP MX v1.0: E8M0 scale per 32 k, E4M3 or E2M1 elements; seeds 971, 972), two
    input sets rotated.  TFLOP/s back to back and per call, like cell()."""
    import torch
    import workloads as wl
    code = {wl.MX_E4M3: g.MX_E4M3, wl.MX_E2M1: g.MX_E2M1}[elem]
    p = wl.mx_problem(971, n, n, n, elem=elem, c_dtype=wl.BF16)
    dev = torch.device("cuda", torch.cuda.current_device())
    sets = [(p.A.to(dev), p.SA.to(dev), p.B.to(dev), p.SB.to(dev), p.C.clone().to(dev)) for _ in range(2)]
    need = g.gemm_mx_workspace_size(n, n, n, code)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)

    def call(i):
        A, SA, B, SB, C = sets[i % 2]
        g.gemm_mx(n, n, n, code, A, p.lda, SA, B, p.ldb, SB, C, n, wl.BF16, 1.0, 0.0, None, wl.EPI_NONE,
                  workspace=ws, workspace_bytes=need, stream=stream)

    for i in range(warmup):
        call(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        call(i)
    e1.record(stream)
    torch.cuda.synchronize()
    total = e0.elapsed_time(e1)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        call(i)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    tf = [p.flops / (ev[i].elapsed_time(ev[i + 1]) * 1e-3) / 1e12 for i in range(steps)]
    med, ci = bootstrap_ci(tf)
    st = g.gemm_device_status()
    if name is not None:
        SAMPLES[name] = [round(x, 2) for x in tf]
    del sets
    torch.cuda.empty_cache()
    return {"tflops": round(p.flops * steps / (total * 1e-3) / 1e12, 1), "ms": round(total / steps, 4),
            "per_call": {"median": round(med, 1), "ci95": [round(ci[0], 1), round(ci[1], 1)]}, "n": steps,
            "status": st}


def q4_prefill_cell(g, stream, M, N=4096, K=4096, steps=20):
    """Prefill with 4-bit weights: gemm_q4 with M rows of x (the tensor-core kernel, W
    dequantised into tensor memory), gemm_q4_ws (the same below Q4_DEQUANT_ROWS rows, W
    expanded once into its workspace and the dense kernel above), the unfused path
    (gemm_q4_dequantize then gemm() in each call) and gemm() on a W dequantised once (the
    dense rate).
    Seeded random codes / scales (as the decode cells), x ~ N(0,1) fp16, fp16 output;
    TFLOP/s back to back."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    gen = torch.Generator(device=dev)
    gen.manual_seed(78)
    wq = torch.randint(-2 ** 31, 2 ** 31 - 1, (N * K // 8,), dtype=torch.int32, device=dev, generator=gen)
    s = (torch.rand(N * K // 64, device=dev, generator=gen) * 3 + 1) * 2.0 ** -10
    sb = torch.stack([s, -8 * s], dim=1).to(torch.float16).reshape(-1)
    x = torch.randn(M * K, device=dev, generator=gen).to(torch.float16)
    y = torch.empty(M * N, dtype=torch.float16, device=dev)
    w_call = torch.empty(N * K, dtype=torch.float16, device=dev)
    w_once = torch.empty(N * K, dtype=torch.float16, device=dev)
    g.gemm_q4_dequantize(N, K, wq, sb, w_once, g.F16, stream=stream)
    ws = _workspace(g, dev)
    q4ws_need = g.gemm_q4_workspace_size(M, N, K, g.F16)
    q4ws = torch.empty(max(q4ws_need, 256), dtype=torch.uint8, device=dev)
    runs = {
        "fused": lambda: g.gemm_q4(M, N, K, g.F16, x, K, wq, sb, y, N, g.F16, 1.0, 0.0, None, g.EPI_NONE,
                                   stream=stream),
        # the public call for long prompts: fused below Q4_DEQUANT_ROWS rows, W expanded once above
        "gemm_q4_ws": lambda: g.gemm_q4_ws(M, N, K, g.F16, x, K, wq, sb, y, N, g.F16, 1.0, 0.0, None, g.EPI_NONE,
                                           workspace=q4ws, workspace_bytes=q4ws_need, stream=stream),
        "dequantize_then_gemm": lambda: (g.gemm_q4_dequantize(N, K, wq, sb, w_call, g.F16, stream=stream),
                                         g.gemm(M, N, K, g.F16, x, K, 1, w_call, 1, K, y, N, g.F16, 1.0, 0.0, None,
                                                g.EPI_NONE, workspace=ws, workspace_bytes=ws.numel(), stream=stream)),
        "gemm_on_dequantized_w": lambda: g.gemm(M, N, K, g.F16, x, K, 1, w_once, 1, K, y, N, g.F16, 1.0, 0.0, None,
                                                g.EPI_NONE, workspace=ws, workspace_bytes=ws.numel(), stream=stream),
    }
    out = {"shape": f"{M}x{N}x{K}"}
    for name, fn in runs.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        out[name] = {"tflops": round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 1), "us": round(ms * 1e3, 2)}
    out["status"] = g.gemm_device_status()
    del wq, sb, x, y, w_call, w_once, q4ws
    torch.cuda.empty_cache()
    return out


def q4_decode_cell(g, stream, M, N=16384, K=16384, reps=50, compact=False):
    """Decode with 4-bit group-quantized weights (gemm_q4): M rows of x against an
    N x K weight matrix, HBM-bound.  Two weight sets (2 x 151 MB > L2) alternate;
    codes and scale/bias are seeded random (uniform codes 0..15, scales in
    [2^-10, 2^-8), biases -8 x scale), x ~ N(0,1) fp16, fp16 output.  Roofline:
    algorithmic bytes (weights + scales + x + y) per call / mean call time,
    against the measured HBM copy bandwidth."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    gen = torch.Generator(device=dev)
    gen.manual_seed(77)
    sets = []
    for _ in range(2):
        wq = torch.randint(-2 ** 31, 2 ** 31 - 1, (N * K // 8,), dtype=torch.int32, device=dev, generator=gen)
        s = (torch.rand(N * K // 64, device=dev, generator=gen) * 3 + 1) * 2.0 ** -10
        sb = torch.stack([s, -8 * s], dim=1).to(torch.float16).reshape(-1)
        x = torch.randn(M * K, device=dev, generator=gen).to(torch.float16)
        sets.append((x, wq, sb, torch.empty(M * N, dtype=torch.float16, device=dev)))

    def call(i):
        x, wq, sb, y = sets[i % 2]
        g.gemm_q4(M, N, K, g.F16, x, K, wq, sb, y, N, g.F16, 1.0, 0.0, None, g.EPI_NONE, stream=stream)

    for i in range(5):
        call(i)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record(stream)
    for i in range(reps):
        call(i)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    st = g.gemm_device_status()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(reps)]
    nbytes = N * K // 2 + (N * K // 64) * 4 + M * K * 2 + M * N * 2
    gbs = [nbytes / (t * 1e-3) / 1e9 for t in per]
    med, ci = bootstrap_ci(gbs)
    mean_ms = ev[0].elapsed_time(ev[reps]) / reps
    achieved = nbytes / (mean_ms * 1e-3) / 1e9
    peak = measured_peaks()["hbm_gbs"]
    del sets
    torch.cuda.empty_cache()
    SAMPLES[f"q4_decode_M{M}"] = [round(x, 1) for x in gbs]
    if compact:
        return {"shape": f"{M}x{N}x{K}", "gbs": round(med, 1), "ci95": [round(ci[0], 1), round(ci[1], 1)],
                "us": round(mean_ms * 1e3, 2), "frac": round(achieved / peak, 4), "n": reps, "status": st}
    return {"M": M, "N": N, "K": K, "bytes_per_call": nbytes, "median_gbs": round(med, 1),
            "ci95": [round(ci[0], 1), round(ci[1], 1)], "mean_us": round(mean_ms * 1e3, 2),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4)},
            "tflops": round(2.0 * M * N * K / (mean_ms * 1e-3) / 1e12, 2), "reps": reps, "status": st}


def alu_fp16_roofline_tflops(num_sms, sm_mhz):
    """Baseline (A) of the cheap-baseline gate: fp16 FMA on the CUDA cores, taken as
    2 x the FP32 FMA rate (128 lanes x 2 halves x 2 flops per SM per clock, HFMA2)."""
    return num_sms * 128 * 2 * 2 * sm_mhz * 1e6 / 1e12


def gate_verdict(tcgen05, alu, simt, mma_sync, win=1.10):
    """Rigel section 3: a kernel wins only if it beats the strongest trivial explanation by >= 1.10x."""
    strongest = max(alu, simt, mma_sync)
    ratio = tcgen05 / strongest
    return {"over_strongest": round(ratio, 3), "over_simt": round(tcgen05 / simt, 2),
            "over_mma_sync": round(tcgen05 / mma_sync, 3), "over_alu_roofline": round(tcgen05 / alu, 2),
            "threshold": win, "win": bool(ratio >= win)}


def baseline_gate(g, stream, l2=L2_BYTES):
    """The cheap-baseline gate (Rigel section 3; section 4, signal 2) on the headline
    workload: the tcgen05 kernel against (A) the CUDA-core fp16 roofline, (B) the
    SIMT kernel and (C) the warp-level mma.sync kernel, all through the C ABI."""
    import torch
    import workloads as wl
    p = wl.fp16_alpha_beta(4096)
    tc = cell(g, p, 30, 5, stream, name="gate_tcgen05", l2=l2)
    simt = cell(g, p, 5, 1, stream, n_sets=2, baseline=g.BASELINE_SIMT, name="gate_simt", l2=l2)
    ms = cell(g, p, 30, 5, stream, baseline=g.BASELINE_MMA_SYNC, name="gate_mma_sync", l2=l2)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    mhz = measured_peaks()["sm_max_mhz"]
    alu = alu_fp16_roofline_tflops(sms, mhz)
    out = {"tcgen05": tc, "simt": simt, "mma_sync": ms, "alu_fp16_roofline_tflops": round(alu, 1)}
    out.update(gate_verdict(tc["tflops"], alu, simt["tflops"], ms["tflops"]))
    return out


# ------------------------------------------------------------ reference arm --

def run_reference(a):
    """The float64 CPU oracle on the host cores, same metric and workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import workloads as wl
    p = wl.fp16_alpha_beta(a.size)
    per_sample = max(1.0, min(a.cpu_seconds / max(1, a.steps + a.warmup), 10.0))
    for _ in range(a.warmup):
        cpu_baseline(p, per_sample, single_sample=True)
    vals, secs = [], 0.0
    t0 = time.perf_counter()
    for _ in range(a.steps):
        r = cpu_baseline(p, per_sample, single_sample=True)
        vals.append(r["value"])
        secs += r["seconds"]
    wall = time.perf_counter() - t0
    value = statistics.median(vals)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = f"each step: 16 random output rows of the {a.size}^3 workload (full K, N), float64 oracle"
    out = {"metric": METRIC, "impl": "reference", "value": value, "unit": "TFLOP/s", "n_gpus": a.gpus,
           "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(1e3 * wall / a.steps, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic: seeded A,B ~ N(0,1)/sqrt(K) fp16, C ~ N(0,1) fp16",
           "config": workload_config(a.size),
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "gpu_launches": 0}
    print(json.dumps(out), flush=True)


def main(argv=None):
    a = _args(argv)
    if a.impl == "reference":
        run_reference(a)
        return
    why = refuse_multi_gpu(a)
    if why:
        print(why, file=sys.stderr, flush=True)
        raise SystemExit(2)
    if a.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if a.profile:
        if a.profile not in PROFILE_CASES:
            raise SystemExit(f"unknown --profile case {a.profile}")
        run_profile(a)
    elif a.q4_decode:
        import torch
        import dense_gemm_epilogues_tcgen05_gb300 as g
        g.gemm_set_q4_kernel({"auto": g.Q4_AUTO, "ffma": g.Q4_FFMA, "mma": g.Q4_MMA}[a.q4_kernel])
        print(json.dumps(q4_decode_cell(g, torch.cuda.current_stream(), a.q4_decode, reps=a.q4_reps)), flush=True)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
