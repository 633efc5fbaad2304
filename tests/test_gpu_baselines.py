"""GPU parity of the cheap-baseline kernels (gemm_baseline): the CUDA-core SIMT
kernel and the warp-level mma.sync kernel compute the same operation as gemm(),
so they meet the same bar against the float64 oracle: integer-valued inputs
(sums < 2^24, exact in fp32 accumulation) bit-exact with fp32 output in every
layout, random workloads within the normalised tolerance, edges never written.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import run_gemm

pytestmark = pytest.mark.gpu

# mma.sync needs the contiguous extents (K, or M / N for M- / N-contiguous operands) to be multiples of 8
SHAPES = [
    (128, 128, 32),      # one tile, one k-slice
    (16, 16, 16),        # far smaller than a tile
    (200, 136, 1000),    # ragged tiles, K not a multiple of the 32-deep slice
    (256, 384, 512),     # several tiles
    (1000, 1000, 1000),
]


def _assert_exact(run):
    y, _ = oracle.gemm_reference(**run.p.oracle_args())
    got = run.values()
    bad = np.argwhere(got != y)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:3].tolist()}: got {got[tuple(bad[0])]} " \
                          f"want {y[tuple(bad[0])]}"


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("ab", [wl.F16, wl.BF16], ids=["f16", "bf16"])
@pytest.mark.parametrize("kind", ["simt", "mma_sync"])
def test_integer_exact_baselines(cuda_lib, kind, ab, layout, shape):
    g = cuda_lib
    M, N, K = shape
    p = wl.random_problem(3000 + M + N + K, M, N, K, ab, wl.F32, layout=layout, alpha=2.0, beta=-1.0,
                          integer=True)
    r = run_gemm(g, p, baseline=g.BASELINE_SIMT if kind == "simt" else g.BASELINE_MMA_SYNC)
    assert r.status == 0
    _assert_exact(r)


@pytest.mark.parametrize("kind", ["simt", "mma_sync"])
@pytest.mark.parametrize("out", [wl.F16, wl.BF16, wl.F32], ids=["f16", "bf16", "f32"])
@pytest.mark.parametrize("epi", [wl.EPI_NONE, wl.EPI_BIAS, wl.EPI_BIAS_GELU, wl.EPI_BIAS_SILU],
                         ids=["none", "bias", "gelu", "silu"])
def test_baseline_epilogues_tolerance(cuda_lib, kind, out, epi):
    g = cuda_lib
    p = wl.random_problem(51, 264, 200, 520, wl.BF16, out, alpha=0.75, beta=0.5 if epi == 0 else 0.0,
                          epilogue=epi)
    r = run_gemm(g, p, baseline=g.BASELINE_SIMT if kind == "simt" else g.BASELINE_MMA_SYNC)
    assert r.status == 0
    res = r.check()
    assert res["pass"], res


def test_mma_sync_fp16_workload(cuda_lib):
    g = cuda_lib
    r = run_gemm(g, wl.fp16_alpha_beta(1024), baseline=g.BASELINE_MMA_SYNC)
    assert r.status == 0
    res = r.check()
    assert res["pass"], res


def test_mma_sync_degenerate_and_rejected(cuda_lib):
    g = cuda_lib
    # K = 0: C = beta * C (as gemm())
    p = wl.random_problem(9, 64, 48, 0, wl.F16, wl.F32, alpha=1.0, beta=0.5)
    r = run_gemm(g, p, baseline=g.BASELINE_MMA_SYNC)
    assert r.status == 0 and r.check()["pass"]
    # an M-contiguous A with M not a multiple of 8 is not taken
    p = wl.random_problem(9, 60, 48, 64, wl.F16, wl.F32, layout="TN", integer=True)
    with pytest.raises(g.GemmError) as e:
        run_gemm(g, p, baseline=g.BASELINE_MMA_SYNC)
    assert e.value.status == g.ERR_UNSUPPORTED
