"""revalidate.py re-derives a bench line's figures from its own data and flags a line whose
recorded figures, gates or record hygiene disagree (no GPU: a synthetic, self-consistent line)."""
import copy
import json
import os
import subprocess
import sys

import numpy as np
import pytest

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
Q4_BYTES = 16384 * 16384 // 2 + (16384 * 16384 // 64) * 4 + 2 * 16384 + 2 * 16384
sys.path.insert(0, REPO)
import revalidate as rv  # noqa: E402


def _line_and_samples():
    rng = np.random.default_rng(5)
    head = list(np.round(1490 + rng.normal(0, 5, 30), 2))
    cell = list(np.round(2680 + rng.normal(0, 8, 30), 2))
    q4 = list(np.round(3207 + rng.normal(0, 3, 50), 1))
    qm, qci = rv.median_and_ci(q4)
    hm, hci = rv.median_and_ci(head)
    cm, cci = rv.median_and_ci(cell)
    M = N = K = 4096
    ms = 0.09341
    value = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    line = {
        "value": round(value, 2), "ms_per_step": ms, "pct_of_nominal_peak": round(100 * value / 2250.0, 2),
        "config": {"M": M, "N": N, "K": K},
        "roofline": {"achieved": round(value, 2), "peak": 1954.3, "frac": round(value / 1954.3, 4)},
        "per_call": {"median_tflops": round(hm, 2), "ci95": [round(hci[0], 2), round(hci[1], 2)]},
        "e2e": {"h2d_bytes_per_step": 3 * 2 * M * N, "d2h_bytes_per_step": 2 * M * N},
        "provenance": {"sources": "x", "recipe_hash": "y", "device": "GB300", "driver": "580", "cuda": "13.0",
                       "torch": "2.9", "cores": 16},
        "clocks": {"reasons": ["sw_power_cap"]},
        "cells": {
            "fp8_4096": {"tflops": 2892.8, "over_fp16": round(2892.8 / 1605.2, 3),
                         "frac_of_2x_bf16_peak": round(2892.8 / (2 * 1954.3), 4),
                         "per_call": {"median": round(cm, 1), "ci95": [round(cci[0], 1), round(cci[1], 1)]}},
            "fp16_twin_4096": {"tflops": 1605.2, "ms": round(2.0 * 4096 ** 3 / 1605.2e12 * 1e3, 4)},
            "q4_decode_M1": {"shape": "1x16384x16384", "gbs": round(qm, 1), "ci95": [round(qci[0], 1), round(qci[1], 1)],
                             "us": 47.64, "frac": round(Q4_BYTES / 47.64e-6 / 1e9 / 6655.6, 4), "n": 50},
            "gelu_M2048": {"fused": {"tflops": 1480.0}, "none": {"tflops": 1534.6}, "decomposed": {"tflops": 980.0},
                           "fused_cost_pct": round(100 * (1534.6 / 1480.0 - 1), 2),
                           "fusion_gain_pct": round(100 * (1480.0 / 980.0 - 1), 2)},
            "baseline_gate_fp16_4096": {"tcgen05": {"tflops": 1532.1}, "simt": {"tflops": 37.4},
                                        "mma_sync": {"tflops": 290.0}, "alu_fp16_roofline_tflops": 161.1,
                                        "over_strongest": round(1532.1 / 290.0, 3), "win": True},
        },
    }
    samples = {"unit": "TFLOP/s per call", "samples": {"headline": head, "fp8_4096": cell, "q4_decode_M1": q4}}
    return line, samples


def _failed(line, samples, peaks={"bf16_tflops": 1954.3, "hbm_gbs": 6655.6}):
    return [c["check"] for c in rv.revalidate(line, samples, peaks).checks if not c["ok"]]


def test_consistent_line_passes():
    line, samples = _line_and_samples()
    assert _failed(line, samples) == []


@pytest.mark.parametrize("mutate,flag", [
    (lambda l, s: l.update(value=l["value"] * 1.02), "value = 2MNK / ms_per_step"),
    (lambda l, s: l["roofline"].update(frac=l["roofline"]["frac"] + 0.01), "roofline.frac = achieved / peak"),
    (lambda l, s: l["per_call"].update(median_tflops=l["per_call"]["median_tflops"] + 10), "headline per-call median"),
    (lambda l, s: s["samples"].update(fp8_4096=[100.0] * 16 + s["samples"]["fp8_4096"][16:]),
     "fp8_4096 per-call median"),
    (lambda l, s: l["cells"]["fp8_4096"].update(over_fp16=1.9), "fp8_4096 over fp16 twin"),
    (lambda l, s: l["cells"]["gelu_M2048"].update(fused_cost_pct=1.0), "gelu_M2048 fused cost %"),
    (lambda l, s: l["cells"]["baseline_gate_fp16_4096"]["tcgen05"].update(tflops=300.0),
     "baseline gate: win at 1.10x"),
    (lambda l, s: l["e2e"].update(h2d_bytes_per_step=0), "e2e h2d bytes per step = A + B + C"),
    (lambda l, s: l["provenance"].pop("recipe_hash"), "provenance complete"),
    (lambda l, s: l["cells"]["fp16_twin_4096"].update(ms=0.09), "fp16_twin_4096 tflops = flops / ms"),
    (lambda l, s: l["cells"]["fp8_4096"].update(frac_of_2x_bf16_peak=0.8), "fp8_4096 frac of 2x bf16 peak"),
    (lambda l, s: l["cells"]["q4_decode_M1"].update(frac=0.6), "q4_decode_M1 frac = bytes / us / HBM peak"),
    (lambda l, s: l["cells"]["q4_decode_M1"].update(gbs=3300.0), "q4_decode_M1 per-call median GB/s"),
    (lambda l, s: l["clocks"]["reasons"].append("hw_slowdown"), "no rejecting throttle reason (clocks)"),
    (lambda l, s: l.update(clocks_cells={"reasons": ["sw_thermal_slowdown"]}),
     "no rejecting throttle reason (clocks_cells)"),
])
def test_each_disagreement_is_flagged(mutate, flag):
    line, samples = _line_and_samples()
    line, samples = copy.deepcopy(line), copy.deepcopy(samples)
    mutate(line, samples)
    assert flag in _failed(line, samples)


def test_command_line_exit_status(tmp_path):
    line, samples = _line_and_samples()
    sp = tmp_path / "samples.json"
    sp.write_text(json.dumps(samples))
    good = tmp_path / "line.json"
    good.write_text("log text\n" + json.dumps(line) + "\n")
    peaks = tmp_path / "peaks.json"
    peaks.write_text(json.dumps({"bf16_tflops": 1954.3}))
    args = [sys.executable, os.path.join(REPO, "revalidate.py"), str(good), "--samples", str(sp), "--peaks", str(peaks)]
    r = subprocess.run(args, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout
    line["value"] *= 1.05
    good.write_text(json.dumps(line) + "\n")
    r = subprocess.run(args, capture_output=True, text=True)
    assert r.returncode == 1 and "value = 2MNK / ms_per_step" in json.loads(r.stdout)["failed"]


def test_gelu_cost_from_rounds_is_the_median_of_paired_ratios():
    """With the rounds recorded, the fused cost is the median over rounds of none_r / fused_r - 1 (each
    round's modes ran side by side): one round with the clock in another state moves the ratio of the
    medians but not this."""
    line, samples = _line_and_samples()
    fused = [1770.0, 1778.0, 1781.0, 1667.0, 1667.0, 1638.0, 1649.0, 1619.0]
    none = [1813.0, 1822.0, 1820.0, 1700.0, 1710.0, 1669.0, 1808.0, 1653.0]
    dec = [x / 1.6 for x in fused]
    paired = float(np.median([100 * (a / b - 1) for a, b in zip(none, fused)]))
    line["cells"]["gelu_M8192"] = {"fused": {"tflops": float(np.median(fused)), "rounds": fused},
                                   "none": {"tflops": float(np.median(none)), "rounds": none},
                                   "decomposed": {"tflops": float(np.median(dec)), "rounds": dec},
                                   "fused_cost_pct": round(paired, 2), "fusion_gain_pct": 60.0}
    assert paired < 3.0 < 100 * (np.median(none) / np.median(fused) - 1)
    assert _failed(line, samples) == []
    line["cells"]["gelu_M8192"]["fused_cost_pct"] = round(100 * (np.median(none) / np.median(fused) - 1), 2)
    assert "gelu_M8192 fused cost %" in _failed(line, samples)
