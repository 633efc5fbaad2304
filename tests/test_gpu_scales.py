"""GPU parity of gemm_ex's product scales (per-tensor alpha_scale read on the
device, per-row and per-column vectors) against the float64 oracle.

Power-of-two scales on integer-valued inputs keep every product and sum exact
in fp32, so those runs must be bit-exact with fp32 output in every kernel
family and orientation: the pair kernel (given and transposed order, one- and
two-pair clusters, whole tiles and stream-K, TMA-staged and direct C stores),
the one-SM kernel, 3xTF32 and the SIMT kernel.  General scales meet the
normalised tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import run_gemm

pytestmark = pytest.mark.gpu


def _assert_exact(run):
    y, _ = oracle.gemm_reference(**run.p.oracle_args())
    got = run.values()
    bad = np.argwhere(got != y)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:3].tolist()}"


@pytest.fixture
def knobs(cuda_lib):
    yield cuda_lib
    cuda_lib.gemm_set_tile_policy(cuda_lib.TILE_AUTO, 0)
    cuda_lib.gemm_set_schedule(cuda_lib.SCHED_AUTO)
    cuda_lib.gemm_set_operand_order(cuda_lib.ORDER_AUTO)
    cuda_lib.gemm_set_multicast(cuda_lib.MCAST_AUTO)


VARIANTS = {
    "pair": dict(policy=3),
    "pair_transposed": dict(policy=3, order=2),
    "pair_given": dict(policy=3, order=1),
    "two_pair_stream_k": dict(policy=3, mcast=2, sched=2),
    "pair_tiles": dict(policy=3, mcast=1, sched=1),
    "one_sm": dict(policy=1),
}


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("ab,out", [(wl.F16, wl.F32), (wl.BF16, wl.F16), (wl.E4M3, wl.F32)],
                         ids=["f16-f32", "bf16-f16", "e4m3-f32"])
def test_integer_exact_scaled(knobs, variant, layout, ab, out):
    g = knobs
    v = VARIANTS[variant]
    g.gemm_set_tile_policy(v["policy"], 0)
    g.gemm_set_operand_order(v.get("order", 0))
    g.gemm_set_multicast(v.get("mcast", 0))
    g.gemm_set_schedule(v.get("sched", 0))
    # integers up to 2 with K = 520: |sum| < 2^11, times scales <= 2^5 -> exact even in fp16 output
    base = wl.random_problem(601, 520, 272, 520, ab, out, layout=layout, alpha=1.0,
                             beta=1.0 if out == wl.F32 else 0.0, integer=True)
    p = wl.with_product_scales(base, 17, dyadic=True)
    if out != wl.F32:
        # keep 16-bit outputs exactly representable: small integer inputs only
        p = wl.with_product_scales(wl.random_problem(602, 136, 264, 64, ab, out, layout=layout, integer=True), 18,
                                   dyadic=True)
    r = run_gemm(g, p)
    assert r.status == 0
    if out == wl.F32:
        _assert_exact(r)
    else:
        y, _ = oracle.gemm_reference(**p.oracle_args())
        want = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float32).to(wl.TORCH_DTYPE[out])
        assert np.array_equal(r.values(), want.to(torch.float64).numpy())


def test_scaled_fp32_paths(knobs):
    """3xTF32 (with a workspace) and the SIMT kernel (without) honour the scales too."""
    g = knobs
    p = wl.with_product_scales(wl.random_problem(71, 200, 136, 96, wl.F32, wl.F32, alpha=2.0, beta=0.5), 19)
    for use_ws in (True, False):
        r = run_gemm(g, p, use_workspace=use_ws)
        assert r.status == 0
        res = r.check()
        assert res["pass"], (use_ws, res)
    # odd ldc: the pair kernel's direct (non-TMA) stores (fp16 output: where beta*C dominates a
    # small scaled product, |z| ~ D and a bf16 output's own rounding would reach the tolerance)
    p = wl.with_product_scales(wl.random_problem(72, 300, 260, 128, wl.BF16, wl.F16, alpha=1.0, beta=1.0, ldc_pad=3,
                                                 epilogue=wl.EPI_BIAS), 20)
    r = run_gemm(g, p)
    res = r.check()
    assert res["pass"], res


@pytest.mark.parametrize("epi", [wl.EPI_NONE, wl.EPI_BIAS_GELU, wl.EPI_BIAS_SILU], ids=["none", "gelu", "silu"])
@pytest.mark.parametrize("out", [wl.F16, wl.BF16, wl.F32], ids=["f16", "bf16", "f32"])
def test_scaled_tolerance(knobs, epi, out):
    g = knobs
    for ab in (wl.F16, wl.E4M3) if out != wl.F16 else (wl.F16,):
        p = wl.with_product_scales(wl.random_problem(81, 1000, 768, 512, ab, out, alpha=0.75,
                                                     beta=0.5 if epi == wl.EPI_NONE else 0.0, epilogue=epi), 21)
        r = run_gemm(g, p)
        res = r.check()
        assert res["pass"], (ab, res)


def test_alpha_scale_is_read_on_the_device(cuda_lib):
    """The same call twice, with only the device value of alpha_scale changed in between."""
    g = cuda_lib
    p = wl.random_problem(91, 256, 256, 128, wl.BF16, wl.F32, integer=True)
    A, B = p.A.cuda(), p.B.cuda()
    s = torch.tensor([1.0], device="cuda")
    outs = []
    for val in (1.0, 4.0):
        s.fill_(val)
        C = torch.zeros(256 * 256, dtype=torch.float32, device="cuda")
        g.gemm_ex(256, 256, 128, wl.BF16, A, p.a_stride_m, p.a_stride_k, B, p.b_stride_k, p.b_stride_n, C, 256,
                  wl.F32, 1.0, 0.0, None, wl.EPI_NONE, alpha_scale=s)
        outs.append(C.cpu())
    assert g.gemm_device_status() == 0
    assert torch.equal(outs[1], 4.0 * outs[0]) and bool(outs[0].abs().sum() > 0)
