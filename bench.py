#!/usr/bin/env python
"""Throughput of the GB300 dense GEMM with fused epilogue.

Headline workload (one "step" = one call of the whole hot path: host dispatch,
tile scheduler, TMA producer, tcgen05 MMA, fused epilogue and store):
    fp16 GEMM M = N = K = 4096, C = 1.5*A*B + 0.5*C, fp16 output, fp32
    accumulation, A, B ~ N(0,1)/sqrt(K), C ~ N(0,1) (seeded, synthetic).
Metric: TFLOP/s (2*M*N*K per step) and % of the GB300 dense tensor peak.

Timing: W untimed warm-up steps, then exactly K steps between a barrier +
device synchronisation on both sides, each step bracketed by CUDA events on
the launch stream.  Three input sets (288 MiB, more than the 129 MB L2) are
used in rotation, so a step does not find its operands in L2.  Under torchrun
every rank runs its own replica (no data-path collective: independent GEMMs),
the time is the max over ranks and ``value`` is the whole job's throughput.

``--impl reference`` times the float64 CPU oracle on the host cores on a
bounded row sample of the same workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
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


def _args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--size", type=int, default=4096)
    ap.add_argument("--no-cells", action="store_true", help="skip the extra per-dtype cells")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle sample budget")
    ap.add_argument("--q4-decode", type=int, default=0, metavar="M",
                    help="only the quantized decode cell with M rows of x (for profiling); prints its JSON")
    ap.add_argument("--q4-reps", type=int, default=50, help="timed calls of the --q4-decode cell")
    ap.add_argument("--q4-kernel", choices=("auto", "ffma", "mma"), default="auto",
                    help="decode kernel of the --q4-decode cell")
    return ap.parse_args(argv)


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
    the job's time is the slowest rank's.  Returns (TFLOP/s, max seconds)."""
    import torch
    world = 1
    t = float(local_seconds)
    if dist is not None and dist.is_initialized():
        world = dist.get_world_size()
        x = torch.tensor([t], dtype=torch.float64, device=device)
        dist.all_reduce(x, op=dist.ReduceOp.MAX)
        t = float(x.item())
    return flops_per_step * steps * world / t / 1e12, t


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


def _make_sets(problem, n_sets, device):
    sets = []
    for _ in range(n_sets):
        sets.append((problem.A.to(device), problem.B.to(device), problem.C.clone().to(device),
                     None if problem.bias is None else problem.bias.to(device)))
    return sets


def _call(g, p, s, stream, baseline=None):
    A, B, C, bias = s
    if baseline is not None:
        g.gemm_baseline(baseline, p.M, p.N, p.K, p.ab_dtype, A, p.a_stride_m, p.a_stride_k, B, p.b_stride_k,
                        p.b_stride_n, C, p.ldc, p.c_dtype, p.alpha, p.beta, bias, p.epilogue, stream=stream)
        return
    ws = _workspace(g, C.device, g.gemm_workspace_size(p.M, p.N, p.K, p.ab_dtype))
    g.gemm(p.M, p.N, p.K, p.ab_dtype, A, p.a_stride_m, p.a_stride_k, B, p.b_stride_k, p.b_stride_n, C, p.ldc,
           p.c_dtype, p.alpha, p.beta, bias, p.epilogue, workspace=ws, workspace_bytes=ws.numel(), stream=stream)


def time_steps(g, p, sets, steps, warmup, stream, sampler=None, dist=None, baseline=None):
    """Warm up, then time `steps` calls; returns (per-step ms list, total ms)."""
    import torch
    for i in range(warmup):
        _call(g, p, sets[i % len(sets)], stream, baseline)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        torch.cuda.synchronize()
        ev[0].record(stream)
        for i in range(steps):
            _call(g, p, sets[i % len(sets)], stream, baseline)
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return per, ev[0].elapsed_time(ev[steps])


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def cell(g, p, steps, warmup, stream, n_sets=3, baseline=None):
    import torch
    sets = _make_sets(p, n_sets, torch.device("cuda", torch.cuda.current_device()))
    per, total = time_steps(g, p, sets, steps, warmup, stream, baseline=baseline)
    tf = [p.flops / (t * 1e-3) / 1e12 for t in per]
    med, ci = bootstrap_ci(tf)
    del sets
    torch.cuda.empty_cache()
    return {"median_tflops": round(med, 1), "ci95": [round(ci[0], 1), round(ci[1], 1)],
            "mean_ms": round(total / steps, 5), "reps": steps}


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
    return {"value": round(p.flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "pipelined": "copy-in / GEMM / copy-out streams, two device buffer sets"}


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
    import torch.distributed as tdist
    import workloads as wl
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        tdist.init_process_group("nccl")
        dist = tdist
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    import dense_gemm_epilogues_tcgen05_gb300 as g

    n = a.size
    p = wl.fp16_alpha_beta(n)
    stream = torch.cuda.current_stream()
    sets = _make_sets(p, 3, dev)
    sampler = ClockSampler(local)
    per, total = time_steps(g, p, sets, a.steps, a.warmup, stream, sampler=sampler, dist=dist)
    st = g.gemm_device_status()
    if st != 0:
        raise RuntimeError(f"device status after timing: {g.gemm_status_string(st)}")
    value, total_s = aggregate(total * 1e-3, p.flops, a.steps, dist, dev)
    tf = [p.flops / (t * 1e-3) / 1e12 for t in per]
    med, ci = bootstrap_ci(tf)
    peaks = measured_peaks()
    avg_ms = sum(per) / len(per)
    achieved = p.flops / (avg_ms * 1e-3) / 1e12
    launch = g.gemm_last_launch()  # what the timed calls enqueued (the same call every step)
    kernel = describe_launch(launch)
    traffic = recorded_traffic("tcgen05_f16_4096")
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": round(total_s * 1e3 / a.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic: seeded A,B ~ N(0,1)/sqrt(K) fp16, C ~ N(0,1) fp16",
        "config": {"workload": WORKLOAD, "M": n, "N": n, "K": n, "layout": "A row-major (K-major), B row-major",
                   "l2": "3 rotating input sets (288 MiB > 129 MB L2)", "parallelism": f"replicas x{world}"},
        "median_tflops": round(med, 2), "ci95": [round(ci[0], 2), round(ci[1], 2)],
        "pct_of_nominal_peak": round(100 * med / NOMINAL_PEAK_TFLOPS["f16"], 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": traffic,
                     "peak_source": f"{peaks['source']} bf16 burst (fp16 runs at the bf16 rate)",
                     "kernel": kernel},
        "clocks": sampler.summary(),
        "gpu_launches": a.steps,
        "launch": launch,
    }
    if rank == 0:
        out["e2e"] = e2e_measure(g, p, 30, stream)
        del sets
        torch.cuda.empty_cache()
        if not a.no_cells and world == 1:
            out["cells"] = extra_cells(g, stream)
        out["cpu_baseline"] = cpu_baseline(p, a.cpu_seconds)
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def extra_cells(g, stream):
    """Per-dtype cells of the headline metric: bf16 and fp8 at 4096^3 (fp8 against
    its fp16 twin), bf16 8192^3, and the cost of the fused bias+GELU epilogue."""
    import workloads as wl
    cells = {}
    cells["bf16_4096_nn"] = cell(g, wl.bf16_nn_large(4096), 30, 5, stream)
    cells["fp8_4096_bf16out"] = cell(g, wl.fp8_e4m3(4096), 30, 5, stream)
    cells["fp16_twin_4096_bf16out"] = cell(g, wl.fp16_twin_of_fp8(4096), 30, 5, stream)
    cells["fp8_over_fp16"] = round(cells["fp8_4096_bf16out"]["median_tflops"] /
                                   cells["fp16_twin_4096_bf16out"]["median_tflops"], 3)
    cells["bf16_8192_nn"] = cell(g, wl.bf16_nn_large(8192), 10, 3, stream, n_sets=2)
    cells["fp32_4096_NN_3xtf32"] = cell(g, wl.fp32_layout("NN", 4096), 20, 3, stream, n_sets=2)
    cells["fp32_4096_TT_3xtf32"] = cell(g, wl.fp32_layout("TT", 4096), 20, 3, stream, n_sets=2)
    for M in (512, 2048, 8192):
        fused = cell(g, wl.bf16_bias_gelu(M), 30, 5, stream)
        plain = cell(g, wl.bf16_bias_gelu(M, epilogue=wl.EPI_NONE), 30, 5, stream)
        cells[f"gelu_M{M}"] = {"fused": fused, "none": plain,
                               "fused_cost_pct": round(100 * (plain["median_tflops"] / fused["median_tflops"] - 1),
                                                       2)}
    cells["baseline_gate_fp16_4096"] = baseline_gate(g, stream)
    for M in (1, 2, 8):
        cells[f"q4_decode_M{M}_16384"] = q4_decode_cell(g, stream, M)
        # the two decode kernels side by side (AUTO above picks one of them)
        for name, kind in (("ffma", g.Q4_FFMA), ("mma", g.Q4_MMA)):
            g.gemm_set_q4_kernel(kind)
            try:
                r = q4_decode_cell(g, stream, M, reps=30)
            finally:
                g.gemm_set_q4_kernel(g.Q4_AUTO)
            cells[f"q4_decode_M{M}_16384"][f"kernel_{name}"] = {k: r[k] for k in ("median_gbs", "ci95", "mean_us")}
    return cells


def q4_decode_cell(g, stream, M, N=16384, K=16384, reps=50):
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


def baseline_gate(g, stream):
    """The cheap-baseline gate (Rigel section 3; section 4, signal 2) on the headline
    workload: the tcgen05 kernel against (A) the CUDA-core fp16 roofline, (B) the
    SIMT kernel and (C) the warp-level mma.sync kernel, all through the C ABI."""
    import torch
    import workloads as wl
    p = wl.fp16_alpha_beta(4096)
    tc = cell(g, p, 30, 5, stream)
    simt = cell(g, p, 5, 1, stream, n_sets=2, baseline=g.BASELINE_SIMT)
    ms = cell(g, p, 30, 5, stream, baseline=g.BASELINE_MMA_SYNC)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    mhz = measured_peaks()["sm_max_mhz"]
    alu = alu_fp16_roofline_tflops(sms, mhz)
    out = {"workload": "fp16 4096^3, C = 1.5*A*B + 0.5*C", "tcgen05": tc, "simt": simt, "mma_sync": ms,
           "alu_fp16_roofline_tflops": round(alu, 1)}
    out.update(gate_verdict(tc["median_tflops"], alu, simt["median_tflops"], ms["median_tflops"]))
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
           "config": {"workload": WORKLOAD, "M": a.size, "N": a.size, "K": a.size,
                      "parallelism": "host cores (oracle)"},
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "gpu_launches": 0}
    print(json.dumps(out), flush=True)


def main(argv=None):
    a = _args(argv)
    if a.warmup < 3 and a.impl == "ours":
        raise SystemExit("--warmup must be >= 3")
    if a.q4_decode:
        import torch
        import dense_gemm_epilogues_tcgen05_gb300 as g
        g.gemm_set_q4_kernel({"auto": g.Q4_AUTO, "ffma": g.Q4_FFMA, "mma": g.Q4_MMA}[a.q4_kernel])
        print(json.dumps(q4_decode_cell(g, torch.cuda.current_stream(), a.q4_decode, reps=a.q4_reps)), flush=True)
    elif a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
