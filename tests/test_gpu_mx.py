"""GPU parity of the block-scaled (MX) product, gemm_mx, against the float64
oracle of the OCP MX v1.0 formats (oracle/mx.py).

Integer-valued elements with scales 2^-1 .. 2^1 keep every product and sum
exact in fp32, so MXFP8 and MXFP4 must match the oracle bit for bit (fp32
outputs; 16-bit outputs as the round-to-nearest-even cast of the exact value)
-- at ragged M, N, K, with a scale drawn per row and block, which pins the
scale layout in tensor memory of both kernels (one SM up to 128 rows of A,
SM pairs beyond).  Quantised normal inputs meet the normalised
tolerance, including the 4096^3 MXFP8 workload on sampled rows.  Guard
canaries around C and its ldc padding must stay intact.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.mx as omx
import workloads as wl
from gpu_util import CANARY, GUARD, sample_rows

pytestmark = pytest.mark.gpu

ELEMS = {"mxfp8": (wl.MX_E4M3, 0), "mxfp4": (wl.MX_E2M1, 1)}


def run_mx(g, p, elem_code, *, workspace_bytes=None):
    view = wl.CODE_VIEW[p.c_dtype]
    n = p.C.numel()
    host = torch.full((2 * GUARD + n,), CANARY[p.c_dtype], dtype=view)
    mid = host[GUARD:GUARD + n]
    mid.copy_(p.C.view(view))
    mid.view(p.M, p.ldc)[:, p.N:] = CANARY[p.c_dtype]
    cbuf = host.cuda()
    c_ptr = cbuf.data_ptr() + GUARD * cbuf.element_size()
    A, SA, B, SB = p.A.cuda(), p.SA.cuda(), p.B.cuda(), p.SB.cuda()
    bias = None if p.bias is None else p.bias.cuda()
    need = g.gemm_mx_workspace_size(p.M, p.N, p.K, elem_code)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    g.gemm_mx(p.M, p.N, p.K, elem_code, A, p.lda, SA, B, p.ldb, SB, c_ptr, p.ldc, p.c_dtype, p.alpha, p.beta,
              bias, p.epilogue, workspace=ws, workspace_bytes=need if workspace_bytes is None else workspace_bytes)
    status = g.gemm_device_status()
    torch.cuda.synchronize()
    back = cbuf.cpu()
    assert bool((back[:GUARD] == CANARY[p.c_dtype]).all()), "guard before C overwritten"
    assert bool((back[GUARD + n:] == CANARY[p.c_dtype]).all()), "guard after C overwritten"
    out = back[GUARD:GUARD + n]
    assert bool((out.view(p.M, p.ldc)[:, p.N:] == CANARY[p.c_dtype]).all()), "ldc padding overwritten"
    return status, out.numpy()


SHAPES = [
    (128, 128, 128),     # one tile, one stage of MXFP8 (one-SM kernel: at most 128 rows)
    (130, 300, 64),      # SM pairs from 129 rows: the peer CTA holds 2 rows, N ends inside B's second block
    (200, 136, 96),      # ragged M and N, K ending inside a stage
    (256, 384, 512),     # several tiles
    (300, 136, 96),      # a second row of pair tiles whose peer half is empty
    (384, 640, 1056),    # K = 33 blocks: a stage with one block
    (1000, 520, 2048),   # many tiles per CTA pair, long K
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("elem", list(ELEMS))
def test_integer_exact(cuda_lib, elem, shape):
    g = cuda_lib
    e, code = ELEMS[elem]
    M, N, K = shape
    p = wl.mx_problem(900 + M + K, M, N, K, elem=e, c_dtype=wl.F32, alpha=1.0, beta=0.0, integer=True)
    st, out = run_mx(g, p, code)
    assert st == 0
    info = g.gemm_last_launch()
    # up to 128 rows one SM per 128 x 256 tile, beyond SM pairs on 256 x 256 tiles
    assert info["path"] == g.PATH_TCGEN05 and info["bn"] == 256
    assert (info["kind"], info["cluster_ctas"]) == ((1, 1) if M <= 128 else (2, 2))
    y, _ = omx.mx_reference(**p.oracle_args())
    got = oracle.output_values(out, p.M, p.N, p.ldc, p.c_dtype)
    bad = np.argwhere(got != y)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:3].tolist()}: got {got[tuple(bad[0])]} " \
                          f"want {y[tuple(bad[0])]}"


@pytest.mark.parametrize("out", [wl.BF16, wl.F16], ids=["bf16", "f16"])
@pytest.mark.parametrize("elem", list(ELEMS))
def test_integer_16bit_outputs_round_exactly(cuda_lib, elem, out):
    g = cuda_lib
    e, code = ELEMS[elem]
    p = wl.mx_problem(951, 264, 392, 384, elem=e, c_dtype=out, integer=True, epilogue=wl.EPI_BIAS_RELU)
    p.bias = torch.round(p.bias * 8)  # integer biases keep the sum exact
    st, got_codes = run_mx(g, p, code)
    assert st == 0
    y, _ = omx.mx_reference(**p.oracle_args())
    want = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float32).to(wl.TORCH_DTYPE[out]).to(torch.float64)
    got = oracle.output_values(got_codes, p.M, p.N, p.ldc, p.c_dtype)
    assert np.array_equal(got, want.numpy())


@pytest.mark.parametrize("epi", [wl.EPI_NONE, wl.EPI_BIAS, wl.EPI_BIAS_GELU, wl.EPI_BIAS_SILU],
                         ids=["none", "bias", "gelu", "silu"])
@pytest.mark.parametrize("out", [wl.BF16, wl.F32], ids=["bf16", "f32"])
@pytest.mark.parametrize("elem", list(ELEMS))
def test_quantised_normal_tolerance(cuda_lib, elem, out, epi):
    g = cuda_lib
    e, code = ELEMS[elem]
    p = wl.mx_problem(961, 1000, 768, 512, elem=e, c_dtype=out, alpha=0.5,
                      beta=0.5 if epi == wl.EPI_NONE else 0.0, epilogue=epi, ldc_pad=8)
    st, got = run_mx(g, p, code)
    assert st == 0
    res = omx.check(p.oracle_args(), got)
    assert res["pass"], res


@pytest.mark.parametrize("elem", list(ELEMS))
def test_4096_workload_sampled_rows(cuda_lib, elem):
    g = cuda_lib
    e, code = ELEMS[elem]
    p = wl.mx_problem(971, 4096, 4096, 4096, elem=e, c_dtype=wl.BF16)
    st, got = run_mx(g, p, code)
    assert st == 0
    res = omx.check(p.oracle_args(), got, rows=sample_rows(4096, n_random=128))
    assert res["pass"], res


def test_alpha_zero_reads_no_operand(cuda_lib):
    g = cuda_lib
    p = wl.mx_problem(981, 130, 70, 64, elem=wl.MX_E4M3, c_dtype=wl.F32, alpha=0.0, beta=2.0, integer=True,
                      epilogue=wl.EPI_BIAS)
    st, got = run_mx(g, p, 0)
    assert st == 0 and g.gemm_last_launch()["path"] == g.PATH_EPILOGUE_ONLY
    res = omx.check(p.oracle_args(), got)  # beta * C + bias in fp32: the fp32 tolerance, not bit equality
    assert res["pass"], res


def test_argument_errors(cuda_lib):
    g = cuda_lib
    p = wl.mx_problem(991, 128, 128, 128, elem=wl.MX_E4M3, c_dtype=wl.F32)
    A, SA, B, SB, C = p.A.cuda(), p.SA.cuda(), p.B.cuda(), p.SB.cuda(), p.C.cuda()
    need = g.gemm_mx_workspace_size(128, 128, 128, g.MX_E4M3)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = (A, 128, SA, B, 128, SB, C, 128, wl.F32, 1.0, 0.0, None, wl.EPI_NONE)
    with pytest.raises(g.GemmError) as ei:  # K not a multiple of the block
        g.gemm_mx(128, 128, 112, g.MX_E4M3, *args, workspace=ws, workspace_bytes=need)
    assert ei.value.status == g.ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as ei:  # workspace too small
        g.gemm_mx(128, 128, 128, g.MX_E4M3, *args, workspace=ws, workspace_bytes=need - 256)
    assert ei.value.status == g.ERR_WORKSPACE
    with pytest.raises(g.GemmError) as ei:  # row pitch not a multiple of 16 bytes
        g.gemm_mx(64, 128, 96, g.MX_E4M3, A, 104, SA, B, 128, SB, C, 128, wl.F32, 1.0, 0.0, None, wl.EPI_NONE,
                  workspace=ws, workspace_bytes=need)
    assert ei.value.status == g.ERR_MISALIGNED
    with pytest.raises(g.GemmError) as ei:  # an fp8 output is not offered here
        g.gemm_mx(128, 128, 128, g.MX_E4M3, A, 128, SA, B, 128, SB, C, 128, wl.E4M3, 1.0, 0.0, None, wl.EPI_NONE,
                  workspace=ws, workspace_bytes=need)
    assert ei.value.status == g.ERR_UNSUPPORTED
    assert g.gemm_device_status() == 0
