"""GPU parity of the 4-bit quantized products (gemm_q4, gemm_q4_dequantize)
against the float64 oracle (oracle.q4), through the C ABI.

* Integer-valued problems (codes 0..15, scale 1 or 2, bias -8..0, x in -2..2:
  every product and partial sum exact in fp32) come back bit-exact with fp32
  output, for every row count 1..8, ragged N and K not a multiple of a warp's
  1024-deep step.
* Realistic problems (N(0, 0.02^2) weights quantized per group, x ~ N(0,1))
  meet the normalised tolerance for every output type and epilogue.
* The full-size decode workloads (1 and 8 x 16384 x 16384) are checked on
  sampled output columns, from the oracle on those weight rows alone.
* Every kernel-dependent test runs on both decode kernels (CUDA-core FFMA and
  tensor-core mma.sync), chosen with gemm_set_q4_kernel.
* The dequantisation pass is exact (rounding of s*q + b, which fp32 holds
  exactly for these inputs), and dequantise-then-gemm() meets the tolerance.
Every call also checks that nothing outside the M x N block of C was written.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import CANARY, GUARD
from oracle import q4

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["ffma", "mma"])
def q4k(request, cuda_lib):
    """Each test runs on both decode kernels: CUDA-core FFMA and tensor-core mma.sync."""
    g = cuda_lib
    g.gemm_set_q4_kernel(g.Q4_FFMA if request.param == "ffma" else g.Q4_MMA)
    yield g
    g.gemm_set_q4_kernel(g.Q4_AUTO)


def run_q4(g, p, workspace=False):
    """Run a Q4Problem on the GPU with guarded C; returns the output codes (M x ldc flat).  With
    `workspace`, through gemm_q4_ws with the workspace it asks for (guarded too)."""
    view = wl.CODE_VIEW[p.c_dtype]
    n = p.C.numel()
    host = torch.full((2 * GUARD + n,), CANARY[p.c_dtype], dtype=view)
    mid = host[GUARD:GUARD + n]
    mid.copy_(p.C.view(view))
    mid.view(p.M, p.ldc)[:, p.N:] = CANARY[p.c_dtype]
    cbuf = host.cuda()
    c_ptr = cbuf.data_ptr() + GUARD * cbuf.element_size()
    X, Wq, SB = p.X.cuda(), p.Wq.cuda(), p.SB.cuda()
    bias = None if p.bias is None else p.bias.cuda()
    if workspace:
        need = g.gemm_q4_workspace_size(p.M, p.N, p.K, p.x_dtype)
        wsb = torch.full((need + 2 * 256,), 0x5A, dtype=torch.uint8, device="cuda")
        g.gemm_q4_ws(p.M, p.N, p.K, p.x_dtype, X, p.ldx, Wq, SB, c_ptr, p.ldc, p.c_dtype, p.alpha, p.beta, bias,
                     p.epilogue, workspace=wsb.data_ptr() + 256, workspace_bytes=need)
        assert g.gemm_device_status() == 0
        back_ws = wsb.cpu()
        assert bool((back_ws[:256] == 0x5A).all()) and bool((back_ws[256 + need:] == 0x5A).all()), "workspace guard"
        run_q4.last_workspace = back_ws[256:256 + need]
    else:
        g.gemm_q4(p.M, p.N, p.K, p.x_dtype, X, p.ldx, Wq, SB, c_ptr, p.ldc, p.c_dtype, p.alpha, p.beta, bias,
                  p.epilogue)
        assert g.gemm_device_status() == 0
    back = cbuf.cpu()
    assert bool((back[:GUARD] == CANARY[p.c_dtype]).all()) and bool((back[GUARD + n:] == CANARY[p.c_dtype]).all())
    out = back[GUARD:GUARD + n]
    assert bool((out.view(p.M, p.ldc)[:, p.N:] == CANARY[p.c_dtype]).all()), "ldc padding overwritten"
    return out.numpy()


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("N,K", [(1, 64), (7, 1088), (64, 1024), (129, 4096), (45, 320)], ids=lambda v: str(v))
@pytest.mark.parametrize("xd", [wl.F16, wl.BF16], ids=["f16", "bf16"])
def test_integer_exact(q4k, M, N, K, xd):
    """Ragged N (a block's 32 rows part-filled), K not a multiple of a stage's 256 k
    (1088, 320: a last stage of one group) or of a warp's 1024-k step."""
    p = wl.q4_problem(100 + M + N + K, M, N, K, xd, wl.F32, integer=True, ldc_pad=3)
    out = run_q4(q4k, p)
    y, _ = q4.q4_reference(**p.oracle_args())
    got = oracle.output_values(out, p.M, p.N, p.ldc, p.c_dtype)
    assert np.array_equal(got, y)


@pytest.mark.parametrize("cd", [wl.F16, wl.BF16, wl.F32], ids=["f16", "bf16", "f32"])
@pytest.mark.parametrize("epi", [wl.EPI_NONE, wl.EPI_BIAS, wl.EPI_BIAS_GELU, wl.EPI_BIAS_SILU],
                         ids=["none", "bias", "gelu", "silu"])
def test_realistic_tolerance(q4k, cd, epi):
    for M, xd in ((1, wl.F16), (4, wl.BF16), (8, wl.F16), (6, wl.BF16)):
        p = wl.q4_problem(7 + M, M, 320, 2048, xd, cd, alpha=1.25, beta=0.5 if epi == wl.EPI_NONE else 0.0,
                          epilogue=epi)
        res = q4.check(p.oracle_args(), run_q4(q4k, p))
        assert res["pass"], (M, res)


def test_degenerate(cuda_lib):
    g = cuda_lib
    # alpha == 0: C = beta*C, weights unread (NULL pointers accepted)
    p = wl.q4_problem(3, 2, 40, 128, wl.F16, wl.F32, alpha=0.0, beta=0.5)
    C = p.C.cuda()
    g.gemm_q4(2, 40, 128, wl.F16, None, 128, None, None, C, p.ldc, wl.F32, 0.0, 0.5, None, wl.EPI_NONE)
    assert g.gemm_device_status() == 0
    y, _ = q4.q4_reference(**p.oracle_args())
    assert np.array_equal(C.cpu().numpy().reshape(2, -1)[:, :40], y.astype(np.float32))


@pytest.mark.parametrize("M", [1, 8])
def test_decode_workload_sampled_columns(q4k, M):
    """M x 16384 x 16384 (the bench's decode cells) on 96 sampled outputs, against the
    oracle run on just those weight rows (an output column needs only its row of W)."""
    N = K = 16384
    p = wl.q4_problem(41, M, N, K, wl.F16, wl.F16)
    out = run_q4(q4k, p)
    rng = np.random.default_rng(7)
    cols = np.unique(np.concatenate([[0, 1, N - 1], rng.integers(0, N, 93)]))
    a = p.oracle_args()
    wq = a["Wq"].reshape(N, K // 8)[cols].reshape(-1)
    sb = a["scale_bias"].reshape(N, K // 64 * 2)[cols].reshape(-1)
    sub = dict(a, N=len(cols), Wq=wq, scale_bias=sb, ldc=len(cols), C=np.zeros(M * len(cols), np.int16))
    y, D = q4.q4_reference(**sub)
    got = oracle.output_values(out, M, N, p.ldc, p.c_dtype)[:, cols]
    err = oracle.max_normalized_error(got, y, D, wl.EPI_NONE)
    assert err <= oracle.tolerance(wl.F16, wl.F16), err


@pytest.mark.parametrize("wd", [wl.F16, wl.BF16], ids=["f16", "bf16"])
def test_dequantize_exact(cuda_lib, wd):
    g = cuda_lib
    p = wl.q4_problem(55, 1, 96, 1024, wd, wd)
    W = torch.empty(96 * 1024, dtype=wl.TORCH_DTYPE[wd], device="cuda")
    g.gemm_q4_dequantize(96, 1024, p.Wq.cuda(), p.SB.cuda(), W, wd)
    assert g.gemm_device_status() == 0
    exact = q4.dequantize(p.Wq.numpy(), p.SB.numpy(), 96, 1024)
    assert np.array_equal(exact.astype(np.float32).astype(np.float64), exact)  # fp32 holds s*q + b exactly
    want = torch.from_numpy(exact).to(torch.float32).to(wl.TORCH_DTYPE[wd]).reshape(-1)
    assert torch.equal(W.cpu().view(torch.int16), want.view(torch.int16))


def test_prefill_dequantize_then_gemm(cuda_lib):
    """Prefill: dequantise to fp16 once, then the dense tensor-core gemm() with W^T as
    B (K-contiguous).  The fp16 rounding of W adds at most 2^-11 of D."""
    g = cuda_lib
    M, N, K = 512, 768, 2048
    p = wl.q4_problem(61, M, N, K, wl.F16, wl.F16, alpha=1.0)
    W = torch.empty(N * K, dtype=torch.float16, device="cuda")
    g.gemm_q4_dequantize(N, K, p.Wq.cuda(), p.SB.cuda(), W, wl.F16)
    C = p.C.clone().cuda()
    g.gemm(M, N, K, wl.F16, p.X.cuda(), K, 1, W, 1, K, C, p.ldc, wl.F16, 1.0, 0.0, None, wl.EPI_NONE)
    assert g.gemm_device_status() == 0
    res = q4.check(p.oracle_args(), C.cpu().view(torch.int16).numpy())
    assert res["pass"], res


# --------------------------------------------------------------- prefill --
# More than 8 rows of x: the tensor-core kernel with W dequantised into tensor
# memory ("X3: Metal GEMM" section 7: the prefill GEMM with the dequantisation
# fused into the multiply-accumulate).


@pytest.mark.parametrize("M,N,K", [(9, 64, 64), (128, 128, 128), (200, 129, 1088), (384, 300, 320),
                                   (1000, 520, 2048)], ids=lambda v: str(v))
@pytest.mark.parametrize("xd", [wl.F16, wl.BF16], ids=["f16", "bf16"])
def test_prefill_integer_exact(cuda_lib, M, N, K, xd):
    """Integer problems (W = s*q + b up to 30, x in -2..2: W exact in 16 bits, sums exact in
    fp32): bit-exact, at ragged M and N (tiles of 128 x 128 part-filled) and K from one group up."""
    g = cuda_lib
    p = wl.q4_problem(300 + M + N + K, M, N, K, xd, wl.F32, integer=True, ldc_pad=5)
    out = run_q4(g, p)
    info = g.gemm_last_launch()
    assert info["path"] == g.PATH_TCGEN05 and info["transposed"] == 1
    y, _ = q4.q4_reference(**p.oracle_args())
    got = oracle.output_values(out, p.M, p.N, p.ldc, p.c_dtype)
    bad = np.argwhere(got != y)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:3].tolist()}: {got[tuple(bad[0])]} vs {y[tuple(bad[0])]}"


@pytest.mark.parametrize("cd", [wl.F16, wl.BF16], ids=["f16", "bf16"])
@pytest.mark.parametrize("epi", [wl.EPI_NONE, wl.EPI_BIAS, wl.EPI_BIAS_GELU, wl.EPI_BIAS_SILU],
                         ids=["none", "bias", "gelu", "silu"])
def test_prefill_realistic_tolerance(cuda_lib, cd, epi):
    """Realistic quantised layers at the 16-bit-output tolerance.  W is rounded to x's 16-bit type
    (at most 2^-11 of |W| for F16 x), which an fp32 output's 1e-5 does not absorb; the fp32 output
    is compared with the unfused path, which rounds W alike (next test)."""
    g = cuda_lib
    for M, xd in ((512, wl.F16), (300, wl.BF16)):
        p = wl.q4_problem(17 + M, M, 768, 2048, xd, cd, alpha=1.25, beta=0.5 if epi == wl.EPI_NONE else 0.0,
                          epilogue=epi)
        res = q4.check(p.oracle_args(), run_q4(g, p))
        assert res["pass"], (M, res)


def test_prefill_matches_dequantize_then_gemm(cuda_lib):
    """The fused prefill and the unfused path (dequantise to fp16, then gemm()) round W alike: their
    outputs agree within fp32 summation order on fp32 outputs."""
    g = cuda_lib
    M, N, K = 640, 512, 4096
    p = wl.q4_problem(62, M, N, K, wl.F16, wl.F32)
    fused = oracle.output_values(run_q4(g, p), M, N, p.ldc, wl.F32)
    W = torch.empty(N * K, dtype=torch.float16, device="cuda")
    g.gemm_q4_dequantize(N, K, p.Wq.cuda(), p.SB.cuda(), W, wl.F16)
    C = torch.zeros(M * N, dtype=torch.float32, device="cuda")
    g.gemm(M, N, K, wl.F16, p.X.cuda(), K, 1, W, 1, K, C, N, wl.F32, 1.0, 0.0, None, wl.EPI_NONE)
    assert g.gemm_device_status() == 0
    unfused = C.cpu().numpy().reshape(M, N).astype(np.float64)
    _, D = q4.q4_reference(**p.oracle_args())
    assert oracle.max_normalized_error(fused, unfused, D, wl.EPI_NONE) <= 1e-5


def test_prefill_large_sampled_rows(cuda_lib):
    """A 4096 x 4096 x 4096 prefill on sampled rows of x."""
    from gpu_util import sample_rows
    g = cuda_lib
    p = wl.q4_problem(71, 4096, 4096, 4096, wl.BF16, wl.BF16)
    out = run_q4(g, p)
    res = q4.check(p.oracle_args(), out, rows=sample_rows(4096, n_random=96))
    assert res["pass"], res


# ------------------------------------------------ long prompts (gemm_q4_ws) --


def _dequantized_w(g, p):
    W = torch.empty(p.N * p.K, dtype=wl.TORCH_DTYPE[p.x_dtype], device="cuda")
    g.gemm_q4_dequantize(p.N, p.K, p.Wq.cuda(), p.SB.cuda(), W, p.x_dtype)
    return W.cpu().view(torch.uint8)


@pytest.mark.parametrize("M,N,K,xd", [(384, 200, 1088, wl.F16), (1000, 520, 2048, wl.BF16)], ids=lambda v: str(v))
def test_q4_ws_integer_exact(cuda_lib, M, N, K, xd):
    """From Q4_DEQUANT_ROWS rows of x with its workspace, gemm_q4_ws expands W once into the workspace
    (its first N*K*2 bytes are then gemm_q4_dequantize's W, byte for byte) and runs the dense kernel:
    bit-exact on integer problems at ragged N, the workspace's guard bytes intact."""
    g = cuda_lib
    p = wl.q4_problem(500 + M + N, M, N, K, xd, wl.F32, integer=True, ldc_pad=3)
    out = run_q4(g, p, workspace=True)
    assert torch.equal(run_q4.last_workspace[:N * K * 2], _dequantized_w(g, p))
    y, _ = q4.q4_reference(**p.oracle_args())
    got = oracle.output_values(out, p.M, p.N, p.ldc, p.c_dtype)
    assert np.array_equal(got, y)


@pytest.mark.parametrize("epi", [wl.EPI_NONE, wl.EPI_BIAS_GELU], ids=["none", "gelu"])
def test_q4_ws_realistic_tolerance_and_fallback(cuda_lib, epi):
    """Realistic layers through gemm_q4_ws meet the 16-bit tolerance at M = 512 (W expanded into the
    workspace, dense kernel) and at M = 64 (below Q4_DEQUANT_ROWS it asks for no workspace and runs the
    fused prefill)."""
    g = cuda_lib
    for M in (512, 64):
        p = wl.q4_problem(520 + M, M, 768, 1024, wl.BF16, wl.BF16, epilogue=epi)
        out = run_q4(g, p, workspace=True)
        if M >= g.Q4_DEQUANT_ROWS:
            assert torch.equal(run_q4.last_workspace[:768 * 1024 * 2], _dequantized_w(g, p))
        else:
            assert run_q4.last_workspace.numel() == 0
        res = q4.check(p.oracle_args(), out)
        assert res["pass"], res
