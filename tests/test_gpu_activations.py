"""GPU parity of the bias + activation epilogues (tanh-form GELU, SiLU, ReLU).

Every kernel family applies the activation: the pair kernel in both operand
orders, the one-SM kernel, the CUDA-core kernel (fp32 inputs, or pitches TMA
cannot take) and the epilogue-only kernel (K = 0).  Random workloads must
meet the normalised tolerance (error scale times max|act'|); the device
activations themselves are checked elementwise over a wide range of z.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import run_gemm

pytestmark = pytest.mark.gpu

NEW_ACTS = [wl.EPI_BIAS_GELU_TANH, wl.EPI_BIAS_SILU, wl.EPI_BIAS_RELU]
ACT_IDS = ["gelu_tanh", "silu", "relu"]
REF = {wl.EPI_BIAS_GELU_TANH: oracle.gelu_tanh, wl.EPI_BIAS_SILU: oracle.silu, wl.EPI_BIAS_RELU: oracle.relu}


@pytest.fixture
def knobs(cuda_lib, request):
    policy, order = request.param
    cuda_lib.gemm_set_tile_policy(policy, 0)
    cuda_lib.gemm_set_operand_order(order)
    yield request.param
    cuda_lib.gemm_set_tile_policy(cuda_lib.TILE_AUTO, 0)
    cuda_lib.gemm_set_operand_order(cuda_lib.ORDER_AUTO)


# (tile policy, operand order): one-SM kernel; pair kernel as given; pair kernel transposed
KNOBS = [(1, 1), (3, 1), (3, 2)]


@pytest.mark.parametrize("knobs", KNOBS, indirect=True, ids=["1sm", "pair", "pair-transposed"])
@pytest.mark.parametrize("out", [wl.F16, wl.BF16, wl.F32], ids=["f16", "bf16", "f32"])
@pytest.mark.parametrize("epi", NEW_ACTS, ids=ACT_IDS)
def test_activation_epilogues_ragged(cuda_lib, epi, out, knobs):
    for ab, layout in ((wl.F16, "NN"), (wl.BF16, "TT"), (wl.E4M3, "NT")):
        if ab == wl.E4M3 and out == wl.F16:
            continue
        p = wl.random_problem(61 + epi, 336, 528, 272, ab, out, layout=layout, alpha=0.8, beta=0.0, epilogue=epi)
        r = run_gemm(cuda_lib, p)
        assert r.status == 0 and r.path == cuda_lib.PATH_TCGEN05
        res = r.check()
        assert res["pass"], (ab, layout, res)


@pytest.mark.parametrize("epi", NEW_ACTS, ids=ACT_IDS)
def test_activation_on_other_kernels(cuda_lib, epi):
    g = cuda_lib
    # fp32 inputs without a workspace: CUDA-core kernel; with one: 3xTF32 pair kernel
    p = wl.random_problem(71, 200, 136, 96, wl.F32, wl.F32, alpha=1.0, beta=0.5, epilogue=epi)
    for use_ws in (False, True):
        r = run_gemm(g, p, use_workspace=use_ws)
        assert r.status == 0
        res = r.check()
        assert res["pass"], (use_ws, res)
    # K = 0: epilogue-only kernel on beta*C + bias
    p0 = wl.random_problem(72, 96, 80, 0, wl.BF16, wl.F32, beta=1.5, epilogue=epi)
    r0 = run_gemm(g, p0)
    assert r0.path == g.PATH_EPILOGUE_ONLY
    assert r0.check()["pass"]
    # misaligned A base: CUDA-core kernel with 16-bit inputs
    p1 = wl.random_problem(73, 144, 160, 64, wl.BF16, wl.BF16, epilogue=epi)
    r1 = run_gemm(g, p1, a_elem_offset=1)
    assert r1.path == g.PATH_SIMT and r1.check()["pass"]


@pytest.mark.parametrize("epi", NEW_ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("ab", [wl.BF16, wl.F32], ids=["tcgen05", "simt"])
def test_activation_accuracy_over_range(cuda_lib, epi, ab):
    """z = bias exactly (the product is zero): fp32 output against the float64 activation."""
    g = cuda_lib
    M, N, K = 128, 4096, 64
    a = torch.zeros(M, K)
    b = torch.zeros(K, N)
    bias = torch.linspace(-30.0, 30.0, N, dtype=torch.float32)
    p = wl.make_problem("act_range", M, N, K, ab, wl.F32, a, b, alpha=1.0, beta=0.0, bias=bias, epilogue=epi)
    r = run_gemm(g, p, use_workspace=False)
    assert r.status == 0
    got = r.values()
    z = bias.double().numpy()
    want = REF[epi](z)[None, :]
    err = np.abs(got - want)
    # the hardware 2^x / reciprocal approximations: ~1e-7 absolute plus ~3e-7 relative
    assert np.all(err <= 2e-7 + 6e-7 * np.abs(z)[None, :]), float((err / (2e-7 + 6e-7 * np.abs(z))).max())
    assert bool(np.all(got[:, z < 0] <= 0.0)) or epi != wl.EPI_BIAS_RELU


ALL_ACTS = [wl.EPI_BIAS_GELU, wl.EPI_BIAS_GELU_TANH, wl.EPI_BIAS_SILU, wl.EPI_BIAS_RELU]
ALL_REF = {**REF, wl.EPI_BIAS_GELU: oracle.gelu}
# How far the low-precision-output forms may stray from the exact activation, as a multiple of
# |z|: erf-GELU through the degree-6 polynomial normal CDF for F16 outputs (1.1e-4 in Phi) and
# through the fitted tanh form for BF16 outputs (1.41e-4 in Phi, plus the hardware tanh's relative
# error of about 2^-11 times 1/2: 3.9e-4), the hardware tanh of the tanh-GELU and SiLU forms
# (relative error about 2^-11, times |z|/2), ReLU exact.
LOW_FORM_BOUND = {(wl.EPI_BIAS_GELU, wl.F16): 1.2e-4, (wl.EPI_BIAS_GELU, wl.BF16): 4e-4,
                  wl.EPI_BIAS_GELU_TANH: 3e-4, wl.EPI_BIAS_SILU: 3e-4, wl.EPI_BIAS_RELU: 0.0}


@pytest.mark.parametrize("epi", ALL_ACTS, ids=["gelu"] + ACT_IDS)
@pytest.mark.parametrize("out", [wl.F16, wl.BF16], ids=["f16", "bf16"])
@pytest.mark.parametrize("kernel", ["tcgen05", "simt"])
def test_low_precision_output_activations_over_range(cuda_lib, epi, out, kernel):
    """z = bias exactly (the product is zero), 16-bit outputs: each output is the exact activation
    rounded to the output type, give or take the form's bound above (and one rounding step for the
    value that bound moves it to).  With fp16 outputs the normalised metric (D = |z|, times
    max|act'|) stays within the 16-bit tolerance everywhere; a bf16 output's own rounding (up to
    2^-8 of the value) exceeds it where the output is close to |z|, whatever the activation."""
    g = cuda_lib
    M, N, K = 128, 4096, 64
    a = torch.zeros(M, K)
    b = torch.zeros(K, N)
    bias = torch.linspace(-12.0, 12.0, N, dtype=torch.float32)
    ab = wl.BF16
    p = wl.make_problem("act_range16", M, N, K, ab, out, a, b, alpha=1.0, beta=0.0, bias=bias, epilogue=epi)
    # a misaligned A base sends the call to the CUDA-core kernel
    r = run_gemm(g, p, use_workspace=False, a_elem_offset=1 if kernel == "simt" else 0)
    assert r.status == 0 and r.path == (g.PATH_SIMT if kernel == "simt" else g.PATH_TCGEN05)
    got = r.values()
    z = bias.double().numpy()
    want = ALL_REF[epi](z)[None, :]
    ulp = 2.0 ** -10 if out == wl.F16 else 2.0 ** -7          # one unit in the last place, relative
    form = LOW_FORM_BOUND[(epi, out)] if epi == wl.EPI_BIAS_GELU else LOW_FORM_BOUND[epi]
    bound = ulp * np.abs(want) + form * np.abs(z)[None, :] + 1e-30
    err = np.abs(got - want)
    assert np.all(err <= bound), float((err / bound).max())
    if out == wl.F16:
        D = np.broadcast_to(np.abs(z)[None, :], got.shape)
        assert oracle.max_normalized_error(got, want, D, epi) <= oracle.tolerance(ab, out)
