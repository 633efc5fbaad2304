"""GPU parity of the pair kernel's transposed operand order (C^T = B^T A^T).

The kernel may run a problem with B's transpose as the MMA's first operand;
TMEM lanes then hold output columns and the epilogue transposes each staged
box back.  Both orders are pinned here against the float64 oracle:

* integer-valued inputs (sums < 2^24, so fp32 accumulation is exact) with
  16-bit outputs must equal the exact result rounded to nearest-even in the
  output type, bit for bit, in every layout, ragged shape and schedule;
* random workloads with alpha, beta*C, bias and GELU must meet the
  normalised tolerance, and the automatic order must agree with both.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import run_gemm

pytestmark = pytest.mark.gpu

ORDERS = {"given": 1, "transposed": 2}
SHAPES = [
    (128, 256, 128),     # one tile
    (16, 16, 16),        # far smaller than a tile
    (336, 208, 1008),    # ragged M, N, K
    (528, 304, 272),     # ragged: M and N not multiples of 32 in either orientation
    (2048, 2048, 256),   # several tiles per CTA
    (1024, 768, 2048),   # long K
]


@pytest.fixture
def order(cuda_lib, request):
    cuda_lib.gemm_set_operand_order(ORDERS[request.param])
    yield request.param
    cuda_lib.gemm_set_operand_order(cuda_lib.ORDER_AUTO)


def _rounded(y, dtype):
    """Exact float64 integers (< 2^24) rounded to nearest-even in the output type."""
    t = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float32).to(wl.TORCH_DTYPE[dtype])
    return t.to(torch.float64).numpy()


def _assert_rounded_exact(run):
    y, _ = oracle.gemm_reference(**run.p.oracle_args())
    want = _rounded(y, run.p.c_dtype)
    got = run.values()
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:3].tolist()}: got {got[tuple(bad[0])]} " \
                          f"want {want[tuple(bad[0])]}"


@pytest.mark.parametrize("order", list(ORDERS), indirect=True)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("ab,out", [(wl.F16, wl.F16), (wl.BF16, wl.BF16), (wl.F16, wl.BF16), (wl.E4M3, wl.BF16)],
                         ids=["f16-f16", "bf16-bf16", "f16-bf16", "e4m3-bf16"])
def test_integer_exact_16bit_out(cuda_lib, ab, out, layout, shape, order):
    M, N, K = shape
    p = wl.random_problem(2000 + M + 3 * N + K, M, N, K, ab, out, layout=layout, alpha=2.0, beta=-1.0,
                          integer=True)
    r = run_gemm(cuda_lib, p)
    assert r.status == 0 and r.path == cuda_lib.PATH_TCGEN05
    _assert_rounded_exact(r)


@pytest.fixture
def stream_k(cuda_lib):
    cuda_lib.gemm_set_schedule(cuda_lib.SCHED_STREAM_K)
    yield
    cuda_lib.gemm_set_schedule(cuda_lib.SCHED_AUTO)


@pytest.mark.parametrize("order", list(ORDERS), indirect=True)
@pytest.mark.parametrize("layout", ["NN", "TT"])
def test_integer_exact_stream_k(cuda_lib, layout, order, stream_k):
    """Every tile split over all SM pairs: partial sums and the owner's epilogue in both orders."""
    for (M, N, K) in [(1024, 1024, 2048), (784, 520, 1536)]:
        p = wl.random_problem(77 + M + N, M, N, K, wl.BF16, wl.BF16, layout=layout, alpha=1.0, beta=1.0,
                              integer=True)
        r = run_gemm(cuda_lib, p)
        assert r.status == 0 and r.path == cuda_lib.PATH_TCGEN05
        _assert_rounded_exact(r)


@pytest.mark.parametrize("order", list(ORDERS), indirect=True)
@pytest.mark.parametrize("out", [wl.F16, wl.BF16], ids=["f16", "bf16"])
@pytest.mark.parametrize("epi", [wl.EPI_NONE, wl.EPI_BIAS, wl.EPI_BIAS_GELU], ids=["none", "bias", "gelu"])
@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_epilogues_ragged(cuda_lib, out, epi, layout, order):
    for ab in (wl.F16, wl.BF16):
        p = wl.random_problem(91, 304, 528, 272, ab, out, layout=layout, alpha=0.75,
                              beta=0.5 if epi == wl.EPI_NONE else 0.0, epilogue=epi)
        r = run_gemm(cuda_lib, p)
        assert r.path == cuda_lib.PATH_TCGEN05
        res = r.check()
        assert res["pass"], res


@pytest.mark.parametrize("order", list(ORDERS), indirect=True)
def test_workloads_both_orders(cuda_lib, order):
    for p in (wl.fp16_alpha_beta(1000), wl.bf16_bias_gelu(512, N=1024, K=768)):
        r = run_gemm(cuda_lib, p)
        assert r.path == cuda_lib.PATH_TCGEN05
        res = r.check()
        assert res["pass"], (p.name, res)


def test_fp32_output_and_padded_ldc_keep_working(cuda_lib):
    """Orders that cannot transpose (fp32 output; C pitch that TMA cannot take) fall back to the given order."""
    g = cuda_lib
    g.gemm_set_operand_order(g.ORDER_TRANSPOSED)
    try:
        for out, pad in ((wl.F32, 0), (wl.BF16, 3)):
            p = wl.random_problem(5, 384, 320, 256, wl.BF16, out, alpha=2.0, beta=-1.0, integer=True, ldc_pad=pad)
            r = run_gemm(g, p)
            assert r.status == 0
            if out == wl.F32:
                y, _ = oracle.gemm_reference(**p.oracle_args())
                assert np.array_equal(r.values(), y)
            else:
                _assert_rounded_exact(r)
    finally:
        g.gemm_set_operand_order(g.ORDER_AUTO)
