"""Re-derive the verdicts of a bench.py line from what the line and its samples file hold.

Rigel section 3 (reporting) pairs every benchmark cell with an independent
re-validator that recomputes pass / fail from the recorded data rather than
trusting the harness that wrote it.  This script is that check for
``bench.py``'s JSON line: it shares no code with ``bench.py`` and recomputes

* the headline: value = 2*M*N*K / ms_per_step, the roofline fraction against
  the measured peak in MEASURED_PEAKS.json, pct of the nominal peak;
* every per-call summary it has samples for: median and the 95 % bootstrap CI
  of the median (10^4 resamples, seed 0, percentile method);
* every cell's rate from its time per call (flops / ms), its fraction of
  twice the bf16 peak where it states one, and each quantized decode cell's
  roofline fraction (algorithmic bytes / time / measured HBM bandwidth) and
  per-call median;
* the derived ratios and gates: fp8 over its fp16 twin (>= 1.5 counts as
  accelerated), fused bias+GELU cost against none and gain against the
  decomposed pass, the cheap-baseline gate (tcgen05 >= 1.10 x the strongest
  baseline), the end-to-end bytes per step of the 4096^3 fp16 workload;
* the record's hygiene: provenance fields present, no throttle reason that
  rejects a run (hw_slowdown, hw_thermal_slowdown, sw_thermal_slowdown).

Usage:  python revalidate.py BENCH_LINE.json [--samples FILE] [--peaks FILE]
Prints one JSON object {"checks": [...], "failed": [...]} and exits 1 when a
recomputed figure disagrees with the line (or a required field is missing).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
NOMINAL_F16_TFLOPS = 2250.0
REJECTING_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")
PROVENANCE_FIELDS = ("sources", "recipe_hash", "device", "driver", "cuda", "torch", "cores")


def median_and_ci(samples, reps=10000, seed=0):
    x = np.sort(np.asarray(samples, dtype=np.float64))
    rng = np.random.default_rng(seed)
    meds = np.median(x[rng.integers(0, x.size, size=(reps, x.size))], axis=1)
    return float(np.median(x)), (float(np.percentile(meds, 2.5)), float(np.percentile(meds, 97.5)))


def cell_flops(name: str):
    """2 M N K of a cell, from its name (None for a cell whose name fixes no GEMM shape)."""
    m = re.fullmatch(r"(?:fp32|fp16|fp8|fp16_twin|bf16|mxfp8|mxfp4)_(\d+)(?:_(?:NN|NT|TN|TT|nn|f32out))?", name)
    if m:
        return 2.0 * int(m.group(1)) ** 3
    m = re.fullmatch(r"gelu_M(\d+)", name)
    if m:
        return 2.0 * int(m.group(1)) * 4096 * 4096
    if name == "baseline_gate_fp16_4096":
        return 2.0 * 4096 ** 3
    return None


def _timed_records(name, cell):
    """(suffix, record) of every timed mode of a cell: the cell itself, or its modes."""
    if "tflops" in cell and "ms" in cell:
        return [("", cell)]
    return [(f".{k}", v) for k, v in cell.items() if isinstance(v, dict) and "tflops" in v and "ms" in v]


class Checker:
    def __init__(self):
        self.checks = []

    def close(self, name, got, want, rel=2e-3, abs_=0.06):
        ok = got is not None and want is not None and math.isfinite(float(got)) and \
            abs(float(got) - float(want)) <= max(abs_, rel * abs(float(want)))
        self.checks.append({"check": name, "recorded": got, "recomputed": want, "ok": bool(ok)})

    def true(self, name, cond, detail=None):
        self.checks.append({"check": name, "ok": bool(cond), **({"detail": detail} if detail is not None else {})})

    def verdict(self, name, recorded, recomputed):
        self.checks.append({"check": name, "recorded": recorded, "recomputed": recomputed,
                            "ok": bool(recorded == recomputed)})


def revalidate(line: dict, samples: dict | None, peaks: dict | None) -> Checker:
    ck = Checker()
    cfg = line.get("config", {})
    M, N, K = cfg.get("M"), cfg.get("N"), cfg.get("K")
    ck.true("config has M, N, K", None not in (M, N, K))
    if None not in (M, N, K) and line.get("ms_per_step"):
        ck.close("value = 2MNK / ms_per_step", line["value"], 2.0 * M * N * K / (line["ms_per_step"] * 1e-3) / 1e12,
                 rel=1e-3)
        ck.close("pct_of_nominal_peak", line.get("pct_of_nominal_peak"), 100 * line["value"] / NOMINAL_F16_TFLOPS)
    roof = line.get("roofline") or {}
    ck.close("roofline.achieved = value", roof.get("achieved"), line["value"])
    if peaks is not None:
        ck.close("roofline.peak = measured bf16 burst", roof.get("peak"), peaks["bf16_tflops"])
    if roof.get("peak"):
        ck.close("roofline.frac = achieved / peak", roof.get("frac"), roof["achieved"] / roof["peak"], rel=1e-3,
                 abs_=1e-3)
    # per-call summaries recomputed from the samples
    if samples is not None:
        got = samples.get("samples", samples)
        if "headline" in got and line.get("per_call"):
            med, ci = median_and_ci(got["headline"])
            ck.close("headline per-call median", line["per_call"]["median_tflops"], med)
            ck.close("headline per-call CI low", line["per_call"]["ci95"][0], ci[0])
            ck.close("headline per-call CI high", line["per_call"]["ci95"][1], ci[1])
        for name, cell in (line.get("cells") or {}).items():
            if isinstance(cell, dict) and name in got and isinstance(cell.get("per_call"), dict):
                med, ci = median_and_ci(got[name])
                ck.close(f"{name} per-call median", cell["per_call"]["median"], med)
                ck.close(f"{name} per-call CI", cell["per_call"]["ci95"][1], ci[1])
    cells = line.get("cells") or {}
    # each cell's rate from its own time per call: tflops = flops / ms (both rounded as recorded)
    for name, cell in cells.items():
        for mode, rec in _timed_records(name, cell):
            flops = cell_flops(name)
            if flops and rec.get("ms"):
                want = flops / (rec["ms"] * 1e-3) / 1e12
                ck.close(f"{name}{mode} tflops = flops / ms", rec["tflops"], want,
                         rel=0.5e-4 / rec["ms"] + 1e-4, abs_=0.06)
        if peaks is not None and "frac_of_2x_bf16_peak" in cell:
            ck.close(f"{name} frac of 2x bf16 peak", cell["frac_of_2x_bf16_peak"],
                     cell["tflops"] / (2 * peaks["bf16_tflops"]), rel=0, abs_=2e-4)
        m = re.fullmatch(r"q4_decode_M(\d+)", name)
        if m and cell.get("us") and peaks is not None and "hbm_gbs" in peaks:
            Mq = int(m.group(1))
            Nq, Kq = (int(v) for v in cell["shape"].split("x")[1:])
            nbytes = Nq * Kq // 2 + (Nq * Kq // 64) * 4 + 2 * Mq * Kq + 2 * Mq * Nq
            ck.close(f"{name} frac = bytes / us / HBM peak", cell["frac"],
                     nbytes / (cell["us"] * 1e-6) / 1e9 / peaks["hbm_gbs"], rel=0, abs_=2e-4)
            if samples is not None and name in samples.get("samples", samples):
                med, ci = median_and_ci(samples.get("samples", samples)[name])
                ck.close(f"{name} per-call median GB/s", cell["gbs"], med)
                ck.close(f"{name} per-call CI", cell["ci95"][1], ci[1])
    # fp8 over the fp16 twin, and the accelerated gate
    for n in (2048, 4096, 8192):
        c8, c16 = cells.get(f"fp8_{n}"), cells.get(f"fp16_twin_{n}")
        if c8 and c16:
            ratio = c8["tflops"] / c16["tflops"]
            ck.close(f"fp8_{n} over fp16 twin", c8.get("over_fp16"), ratio, abs_=2e-3)
            ck.checks.append({"check": f"fp8_{n} accelerated (>= 1.5x fp16)", "recomputed": ratio >= 1.5, "ok": True})
    # fused bias+GELU: the median over rounds of the ratio of the rates taken side by side in a
    # round (with the rounds recorded), else the ratio of the modes' rates
    def paired(num, den):
        if num.get("rounds") and den.get("rounds"):
            return float(np.median([100 * (a / b - 1) for a, b in zip(num["rounds"], den["rounds"])]))
        return 100 * (num["tflops"] / den["tflops"] - 1)
    for M_ in (512, 2048, 8192):
        c = cells.get(f"gelu_M{M_}")
        if c:
            cost = paired(c["none"], c["fused"])
            ck.close(f"gelu_M{M_} fused cost %", c["fused_cost_pct"], cost, abs_=0.02)
            ck.close(f"gelu_M{M_} fusion gain %", c["fusion_gain_pct"], paired(c["fused"], c["decomposed"]),
                     abs_=0.02)
            ck.checks.append({"check": f"gelu_M{M_} fused cost <= 5 %", "recomputed": cost <= 5.0, "ok": True})
    # cheap-baseline gate
    gate = cells.get("baseline_gate_fp16_4096")
    if gate:
        strongest = max(gate["simt"]["tflops"], gate["mma_sync"]["tflops"], gate["alu_fp16_roofline_tflops"])
        ratio = gate["tcgen05"]["tflops"] / strongest
        ck.close("baseline gate: over the strongest baseline", gate["over_strongest"], ratio, abs_=2e-3)
        ck.verdict("baseline gate: win at 1.10x", gate["win"], ratio >= 1.10)
    # end-to-end bytes of the headline workload (fp16 A, B, C in; C out)
    e2e = line.get("e2e") or {}
    if None not in (M, N, K) and e2e:
        ck.verdict("e2e h2d bytes per step = A + B + C", e2e.get("h2d_bytes_per_step"), 2 * (M * K + K * N + M * N))
        ck.verdict("e2e d2h bytes per step = C", e2e.get("d2h_bytes_per_step"), 2 * M * N)
    # hygiene
    prov = line.get("provenance") or {}
    missing = [f for f in PROVENANCE_FIELDS if not prov.get(f)]
    ck.true("provenance complete", not missing, detail=missing or None)
    for key in ("clocks", "clocks_cells"):
        if key == "clocks" or key in line:
            reasons = (line.get(key) or {}).get("reasons") or []
            bad = [r for r in reasons if any(r.startswith(x) for x in REJECTING_REASONS)]
            ck.true(f"no rejecting throttle reason ({key})", not bad, detail=bad or None)
    return ck


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("line", help="file holding bench.py's JSON line (the last JSON line in it is used)")
    ap.add_argument("--samples", default=None, help="per-call samples file (default: the line's samples_file)")
    ap.add_argument("--peaks", default=os.path.join(HERE, "MEASURED_PEAKS.json"))
    a = ap.parse_args(argv)
    with open(a.line) as f:
        lines = [ln for ln in f.read().splitlines() if ln.strip().startswith("{")]
    line = json.loads(lines[-1])
    spath = a.samples or (os.path.join(HERE, line["samples_file"]) if line.get("samples_file") else None)
    samples = None
    if spath and os.path.exists(spath):
        with open(spath) as f:
            samples = json.load(f)
    peaks = None
    if a.peaks and os.path.exists(a.peaks):
        with open(a.peaks) as f:
            peaks = json.load(f)
    ck = revalidate(line, samples, peaks)
    failed = [c["check"] for c in ck.checks if not c["ok"]]
    print(json.dumps({"checks": ck.checks, "failed": failed}))
    return 1 if failed else 0


if __name__ == "__main__":
    sys.exit(main())
