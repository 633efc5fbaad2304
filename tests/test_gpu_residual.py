"""GPU parity of the post-activation residual (gemm_ex): y = act(z) + R.

The residual is one more input of the pluggable epilogue ("Case Study: Steel's
BlockMMA", the paragraph on the ending where fusion plugs in), read in the
output type and added after the activation.  On integer-valued inputs with
ReLU (exact in fp32) every kernel family must match the float64 oracle bit
for bit -- fp32 outputs exactly, 16-bit outputs as the round-to-nearest-even
cast of the exact value -- while R's padding columns hold NaN that must never
be read: the pair kernel in given and transposed order, one- and two-pair
clusters, whole tiles and stream-K, TMA-staged and direct stores, the one-SM
kernel, 3xTF32, the SIMT kernel and the epilogue-only path.  Random
workloads with GELU meet the normalised tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import run_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture
def knobs(cuda_lib):
    yield cuda_lib
    cuda_lib.gemm_set_tile_policy(cuda_lib.TILE_AUTO, 0)
    cuda_lib.gemm_set_schedule(cuda_lib.SCHED_AUTO)
    cuda_lib.gemm_set_operand_order(cuda_lib.ORDER_AUTO)
    cuda_lib.gemm_set_multicast(cuda_lib.MCAST_AUTO)


def _assert_matches(run):
    """Exact for fp32 outputs; for 16-bit outputs, the RNE cast of the exact (fp32-representable) value."""
    p = run.p
    y, _ = oracle.gemm_reference(**p.oracle_args())
    got = run.values()
    assert not np.isnan(got).any(), "NaN in the output: the residual's padding was read"
    if p.c_dtype == wl.F32:
        want = y
    else:
        want = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float32).to(wl.TORCH_DTYPE[p.c_dtype])
        want = want.to(torch.float64).numpy()
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:3].tolist()}: got {got[tuple(bad[0])]} " \
                          f"want {want[tuple(bad[0])]}"


VARIANTS = {
    "pair": dict(policy=3),
    "pair_transposed": dict(policy=3, order=2),
    "pair_given": dict(policy=3, order=1),
    "two_pair_stream_k": dict(policy=3, mcast=2, sched=2),
    "pair_stream_k": dict(policy=3, mcast=1, sched=2),
    "pair_tiles": dict(policy=3, mcast=1, sched=1),
    "one_sm_256": dict(policy=1),
    "one_sm_128": dict(policy=2),
}


def _set(g, v):
    g.gemm_set_tile_policy(v["policy"], 0)
    g.gemm_set_operand_order(v.get("order", 0))
    g.gemm_set_multicast(v.get("mcast", 0))
    g.gemm_set_schedule(v.get("sched", 0))


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("layout", ["NN", "NT", "TT"])
@pytest.mark.parametrize("ab,out", [(wl.F16, wl.F32), (wl.BF16, wl.BF16), (wl.F16, wl.F16), (wl.E4M3, wl.F32)],
                         ids=["f16-f32", "bf16-bf16", "f16-f16", "e4m3-f32"])
def test_integer_exact_residual(knobs, variant, layout, ab, out):
    g = knobs
    _set(g, VARIANTS[variant])
    # ragged M and N (box and chunk edges; pitches stay multiples of 16 bytes so every layout is
    # TMA-streamed), K long enough for stream-K to split tiles
    base = wl.random_problem(701, 528, 272, 1024, ab, out, layout=layout, alpha=1.0, beta=1.0, integer=True,
                             epilogue=wl.EPI_BIAS_RELU)
    p = wl.with_residual(base, 17, pad=8, integer=True)
    r = run_gemm(g, p)
    assert r.status == 0 and r.path == g.PATH_TCGEN05
    if VARIANTS[variant].get("order") == 2 and out != wl.F32:
        assert g.gemm_last_launch()["transposed"] == 1
    _assert_matches(r)


def test_residual_with_product_scales(knobs):
    g = knobs
    for v in ("pair", "pair_transposed", "two_pair_stream_k"):
        _set(g, VARIANTS[v])
        p = wl.with_residual(wl.with_product_scales(
            wl.random_problem(705, 264, 512, 256, wl.BF16, wl.BF16, integer=True, epilogue=wl.EPI_BIAS_RELU), 23,
            dyadic=True), 24, pad=16, integer=True)
        r = run_gemm(g, p)
        assert r.status == 0
        _assert_matches(r)


def test_residual_fp32_paths(knobs):
    """3xTF32 (with a workspace) and the SIMT kernel (without): exact on integer inputs."""
    g = knobs
    p = wl.with_residual(wl.random_problem(711, 300, 200, 96, wl.F32, wl.F32, alpha=2.0, beta=0.5, integer=True,
                                           epilogue=wl.EPI_BIAS_RELU), 25, pad=5, integer=True)
    for use_ws in (True, False):
        r = run_gemm(g, p, use_workspace=use_ws)
        assert r.status == 0
        assert g.gemm_last_launch()["tf32x3"] == (1 if use_ws else 0)
        _assert_matches(r)


@pytest.mark.parametrize("case", ["odd_ldc", "odd_ldr", "amax", "misaligned_a"])
def test_residual_direct_stores(knobs, case):
    """Outputs that cannot move through shared memory by TMA (odd pitch, or the amax reduction) and a
    residual whose pitch rules out 16-byte loads take the direct stores; the SIMT kernel when A is
    misaligned."""
    g = knobs
    ldc_pad = 3 if case == "odd_ldc" else 0
    base = wl.random_problem(721, 392, 328, 192, wl.BF16, wl.F16, alpha=1.0, beta=1.0, integer=True,
                             ldc_pad=ldc_pad, epilogue=wl.EPI_BIAS_RELU)
    p = wl.with_residual(base, 26, pad=3 if case == "odd_ldr" else 8, integer=True)
    extra = {}
    if case == "amax":
        extra["amax"] = torch.zeros(1, device="cuda")
    r = run_gemm(g, p, extra=extra, a_elem_offset=1 if case == "misaligned_a" else 0)
    assert r.status == 0
    if case == "misaligned_a":
        assert r.path == g.PATH_SIMT
    _assert_matches(r)
    if case == "amax":
        y, _ = oracle.gemm_reference(**p.oracle_args())
        assert float(extra["amax"].item()) == float(np.abs(y).max())


def test_residual_epilogue_only(cuda_lib):
    """K == 0: y = act(beta*C + bias) + R, A and B unread."""
    g = cuda_lib
    p = wl.with_residual(wl.random_problem(731, 130, 70, 0, wl.BF16, wl.F32, alpha=1.0, beta=2.0, integer=True,
                                           epilogue=wl.EPI_BIAS_RELU), 27, pad=2, integer=True)
    r = run_gemm(g, p)
    assert r.status == 0 and r.path == g.PATH_EPILOGUE_ONLY
    _assert_matches(r)


@pytest.mark.parametrize("epi", [wl.EPI_NONE, wl.EPI_BIAS_GELU], ids=["none", "gelu"])
@pytest.mark.parametrize("out", [wl.BF16, wl.F16, wl.F32], ids=["bf16", "f16", "f32"])
def test_residual_tolerance(knobs, epi, out):
    g = knobs
    p = wl.with_residual(wl.random_problem(741, 1000, 768, 512, wl.BF16 if out != wl.F16 else wl.F16, out,
                                           alpha=0.75, beta=0.5 if epi == wl.EPI_NONE else 0.0, epilogue=epi),
                         28, pad=24)
    r = run_gemm(g, p)
    assert r.status == 0
    res = r.check()
    assert res["pass"], res


def test_residual_rejections(cuda_lib):
    g = cuda_lib
    p = wl.random_problem(751, 64, 64, 64, wl.BF16, wl.BF16)
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    R = torch.zeros(64 * 64, dtype=torch.bfloat16, device="cuda")
    args = (64, 64, 64, wl.BF16, A, p.a_stride_m, p.a_stride_k, B, p.b_stride_k, p.b_stride_n)
    with pytest.raises(g.GemmError) as ei:  # ldr < N
        g.gemm_ex(*args, C, 64, wl.BF16, 1.0, 0.0, None, wl.EPI_NONE, residual=R, ldr=63)
    assert ei.value.status == g.ERR_INVALID_ARG
    C8 = torch.zeros(64 * 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(g.GemmError) as ei:  # no residual with an E4M3 output
        g.gemm_ex(*args, C8, 64, wl.E4M3, 1.0, 0.0, None, wl.EPI_NONE, residual=R, ldr=64)
    assert ei.value.status == g.ERR_UNSUPPORTED
