"""bench.py host logic (CPU only): statistics, clock records, traffic lookup,
the reference arm's JSON line, and the multi-rank aggregation under gloo."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

from conftest import REPO

sys.path.insert(0, REPO)
import bench  # noqa: E402


def test_bootstrap_ci_brackets_the_median():
    rng = np.random.default_rng(1)
    x = rng.normal(100.0, 1.0, size=300)
    med, (lo, hi) = bench.bootstrap_ci(x)
    assert med == pytest.approx(float(np.median(x)))
    assert lo <= med <= hi and hi - lo < 0.5
    # fixed seed: the same samples give the same interval
    assert bench.bootstrap_ci(x) == (med, [lo, hi])


def test_bootstrap_ci_bimodal_is_wide():
    x = np.concatenate([np.full(145, 4.65), np.full(155, 6.5)])
    med, (lo, hi) = bench.bootstrap_ci(x)
    assert lo < 5.0 < hi or (lo == hi == 6.5)


def test_clock_record_parsing():
    text = "\n".join([
        "2070, 2070, 120.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "1890, 2070, 1200.0, 0x4, Not Active, Not Active, Not Active, Active",
        "1900, 2070, 1250.0, 0x4, Not Active, Not Active, Not Active, Active",
        "garbage line",
    ])
    s = bench.ClockSampler.parse(text)
    assert s["sm_max_mhz"] == 2070.0
    assert s["sm_mhz"] == pytest.approx(1895.0)   # median of the samples under load
    assert s["reasons"] == ["sw_power_cap"]
    bad = bench.ClockSampler.parse("1500, 2070, 900, 0x8, Active, Not Active, Not Active, Not Active")
    assert "hw_slowdown" in bad["reasons"]


def test_clock_sampler_around_a_region_without_nvidia_smi(monkeypatch):
    """The sampler wraps a region whatever the host has: without nvidia-smi it says so."""
    monkeypatch.setenv("PATH", "/nonexistent")
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    sampler = bench.ClockSampler(0)
    with sampler:
        done = sum(range(1000))
    assert done == 499500
    assert sampler.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}


def test_measured_peaks_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "REPO", str(tmp_path))
    p = bench.measured_peaks()
    assert p["source"] == "fallback" and p["bf16_tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"bf16_tflops": 1954.3, "bf16_tflops_sustained": 1749.8, "hbm_gbs": 6655.6}))
    p = bench.measured_peaks()
    assert p["source"] == "measured" and p["bf16_tflops"] == 1954.3


def test_traffic_record_matches_only_current_sources(tmp_path, monkeypatch):
    import __graft_entry__
    fp = __graft_entry__.build_module().source_fingerprint()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.tsv").write_text(
        f"# comment\n0000000000000000\ttagA\t1\told kernel\n{fp}\ttagA\t12345\tnow\n")
    monkeypatch.setattr(bench, "REPO", str(tmp_path))
    assert bench.recorded_traffic("tagA") == 12345.0
    assert bench.recorded_traffic("tagB") is None


def test_aggregate_single_rank():
    v, t = bench.aggregate(2.0, 1e12, 10)
    assert t == 2.0 and v == pytest.approx(5.0)


def _agg_worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    v, t = bench.aggregate(1.0 + rank, 1e12, 4, dist)
    out[rank] = (v, t)
    dist.destroy_process_group()


def test_aggregate_two_ranks_takes_the_slowest():
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_agg_worker, args=(2, port, out), nprocs=2, join=True)
    for r in range(2):
        v, t = out[r]
        assert t == 2.0                       # max over ranks
        assert v == pytest.approx(2 * 4 * 1e12 / 2.0 / 1e12)  # both ranks' work over that time


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(REPO, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1", "--size", "256", "--cpu-seconds", "1"],
                       capture_output=True, text=True, timeout=300, cwd=REPO)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "config", "cpu_baseline", "e2e", "impl"):
        assert key in line, key
    assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0


def test_describe_launch():
    import bench
    pair = {"path": 2, "kind": 2, "bn": 256, "transposed": 1, "cluster_ctas": 4, "grid_ctas": 144, "tiles": 128,
            "stream_k_tiles": 56, "tf32x3": 0}
    d = bench.describe_launch(pair)
    assert "256x256" in d and "two-pair clusters" in d and "144 CTAs" in d and "C^T" in d and "56 of 128" in d
    one = dict(pair, kind=1, bn=128, cluster_ctas=1, grid_ctas=152, transposed=0, stream_k_tiles=0)
    assert bench.describe_launch(one) == "gemm_tcgen05_kernel 128x128 tiles, 152 CTAs"
    assert bench.describe_launch({"path": 3, "kind": 0}) == "path 3"


def test_baseline_gate_arithmetic():
    import bench
    # 152 SMs at 2070 MHz: 152 * 512 flop/clk * 2.07e9 = 161.1 TFLOP/s
    assert abs(bench.alu_fp16_roofline_tflops(152, 2070.0) - 161.1) < 0.1
    v = bench.gate_verdict(1400.0, 161.1, 30.0, 1000.0)
    assert v["over_strongest"] == 1.4 and v["win"] is True and v["over_mma_sync"] == 1.4
    v = bench.gate_verdict(1050.0, 161.1, 30.0, 1000.0)
    assert v["win"] is False and v["over_strongest"] == 1.05
    # the strongest explanation may be the roofline itself
    assert bench.gate_verdict(170.0, 161.1, 30.0, 100.0)["over_strongest"] == round(170.0 / 161.1, 3)


def test_bench_refuses_more_than_one_gpu():
    """The library is single-GPU (the pair kernel's TMA multicast is for single-GPU processes):
    bench.py exits with an error for --gpus 2 or a multi-rank launch, before touching a GPU."""
    for argv, env in ((["--gpus", "2"], {}), (["--gpus", "1"], {"WORLD_SIZE": "2", "RANK": "0"})):
        r = subprocess.run([sys.executable, os.path.join(REPO, "bench.py"), "--steps", "3", "--warmup", "3"] + argv,
                           capture_output=True, text=True, timeout=120, cwd=REPO, env=dict(os.environ, **env))
        assert r.returncode == 2, (r.returncode, r.stderr)
        assert "one GPU" in r.stderr and r.stdout.strip() == ""
    a = bench._args(["--gpus", "1"])
    assert bench.refuse_multi_gpu(a, env={}) is None
    assert bench.refuse_multi_gpu(a, env={"WORLD_SIZE": "4"}) is not None


def test_bench_has_no_collective_backend():
    """No NCCL process group: nothing in the timed path talks to another GPU."""
    text = open(os.path.join(REPO, "bench.py")).read()
    assert 'init_process_group("nccl")' not in text and "init_process_group('nccl')" not in text


def test_bimodality_flags_two_clock_states():
    rng = np.random.default_rng(3)
    two = np.concatenate([rng.normal(4.65, 0.05, 145), rng.normal(6.5, 0.05, 155)])
    r = bench.bimodality(two)
    assert r["bimodal"] and r["modes"][0] == pytest.approx(4.65, abs=0.05) and r["share"][0] == pytest.approx(
        145 / 300, abs=0.01)
    assert not bench.bimodality(rng.normal(100.0, 1.0, 300))["bimodal"]
    # a few stragglers (under 5 %) are not a second mode
    assert not bench.bimodality(np.concatenate([rng.normal(100, 0.5, 295), [60.0] * 5]))["bimodal"]


def test_reference_arm_shares_the_workload_config():
    r = subprocess.run([sys.executable, os.path.join(REPO, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1", "--size", "256", "--cpu-seconds", "1"],
                       capture_output=True, text=True, timeout=300, cwd=REPO)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["config"] == bench.workload_config(256)


def test_cells_rotate_inputs_beyond_l2():
    import workloads as wl
    p = wl.fp16_alpha_beta(512)
    n = bench.sets_beyond_l2(p, l2_bytes=129 * 10 ** 6)
    assert n * bench.set_bytes(p) > 129 * 10 ** 6
    assert bench.sets_beyond_l2(wl.fp32_square(256)) >= 2


def test_paired_cost_is_robust_to_clock_drift_between_rounds():
    """The fused cost is the median over rounds of none_r / fused_r - 1: a round in which the plain GEMM
    ran in a faster clock state than its fused partner moves one ratio, not the result, while the ratio
    of the two medians moves with it."""
    fused = [1770.0, 1778.0, 1781.0, 1667.0, 1667.0, 1638.0, 1649.0, 1619.0]
    none = [f * 1.02 for f in fused]
    assert abs(bench.paired_pct(none, fused) - 2.0) < 1e-9
    none[6] = 1808.0  # one round of the plain GEMM in the fast state
    assert abs(bench.paired_pct(none, fused) - 2.0) < 1e-9
    assert 100 * (np.median(none) / np.median(fused) - 1) > 2.5
