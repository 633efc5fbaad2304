"""GPU parity of gemm_ex's fp8 E4M3 output (y / out_scale, rounded to nearest
even, saturated at 448) and its amax reduction (max |y| over the outputs),
against the float64 oracle.

* Integer-valued problems (every output exact in fp32, out_scale a power of
  two) must give the round-to-nearest-even, saturating E4M3 code of the exact
  value, and their amax exactly, on every kernel path an
  fp8 output can take: the pair kernel (one- and two-pair clusters, whole
  tiles and stream-K), the SIMT kernel (strides TMA cannot take) and the
  epilogue-only kernel (alpha == 0).
* The fp8 workload (per-tensor quantised E4M3 inputs) with an fp8 output
  scaled by its own amax passes the fp8-output check; amax alone also works
  with 16-bit and fp32 outputs (3xTF32 and SIMT included).
Guards around C and its ldc padding must stay intact.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

GUARD = 64
CANARY8 = 0x5A


def run_ex(g, p, *, out_scale=None, amax=True, use_workspace=True, a_offset=0):
    """gemm_ex on problem p (c_dtype may be E4M3); returns (output codes, amax or None)."""
    dev = "cuda"
    if p.c_dtype == wl.E4M3:
        n = p.M * p.ldc
        host = torch.full((2 * GUARD + n,), CANARY8, dtype=torch.uint8)
        host[GUARD:GUARD + n].view(p.M, p.ldc)[:, :p.N] = 0
    else:
        view = wl.CODE_VIEW[p.c_dtype]
        n = p.C.numel()
        host = torch.zeros((2 * GUARD + n,), dtype=view)
        host[GUARD:GUARD + n] = p.C.view(view)
    cbuf = host.to(dev)
    c_ptr = cbuf.data_ptr() + GUARD * cbuf.element_size()
    A = p.A.to(dev)
    if a_offset:
        big = torch.zeros(A.numel() + a_offset, dtype=A.dtype, device=dev)
        big[a_offset:] = A
        A = big[a_offset:]
    B = p.B.to(dev)
    bias = None if p.bias is None else p.bias.to(dev)
    sc = {k: v.to(dev) for k, v in p.product_scales.items()}
    am = torch.zeros(1, dtype=torch.float32, device=dev) if amax else None
    os_t = None if out_scale is None else torch.tensor([out_scale], dtype=torch.float32, device=dev)
    ws = torch.empty(max(g.gemm_workspace_size(p.M, p.N, p.K, p.ab_dtype), 256), dtype=torch.uint8, device=dev)
    g.gemm_ex(p.M, p.N, p.K, p.ab_dtype, A, p.a_stride_m, p.a_stride_k, B, p.b_stride_k, p.b_stride_n, c_ptr, p.ldc,
              p.c_dtype, p.alpha, p.beta, bias, p.epilogue, out_scale=os_t, amax=am,
              workspace=ws if use_workspace else None, workspace_bytes=ws.numel() if use_workspace else 0, **sc)
    assert g.gemm_device_status() == 0
    back = cbuf.cpu()
    if p.c_dtype == wl.E4M3:
        assert bool((back[:GUARD] == CANARY8).all()) and bool((back[GUARD + n:] == CANARY8).all())
        assert bool((back[GUARD:GUARD + n].view(p.M, p.ldc)[:, p.N:] == CANARY8).all()), "ldc padding written"
    out = back[GUARD:GUARD + n].numpy()
    return out, (None if am is None else float(am.cpu()[0]))


def _fp8_problem(seed, M, N, K, ab, *, layout="NN", alpha=1.0, epilogue=wl.EPI_NONE, ldc_pad=0):
    """Operands in {-1, 0, 1} and integer biases: every y is an integer exact in fp32, so the
    kernel's y / out_scale (a power of two) is the exact quotient and its E4M3 code is the
    round-to-nearest-even, saturating code of the exact value -- the same on both sides."""
    g = torch.Generator().manual_seed(seed)
    a = torch.randint(-1, 2, (M, K), generator=g).to(torch.float32)
    b = torch.randint(-1, 2, (K, N), generator=g).to(torch.float32)
    bias = None if epilogue == wl.EPI_NONE else torch.randint(-2, 3, (N,), generator=g).to(torch.float32)
    q = wl.make_problem(f"fp8out_s{seed}_{M}x{N}x{K}", M, N, K, ab, wl.F32, a, b, None, layout=layout,
                        ldc=N + ldc_pad, alpha=alpha, bias=bias, epilogue=epilogue)
    return wl.dataclasses.replace(q, c_dtype=wl.E4M3, C=torch.zeros(M * (N + ldc_pad), dtype=torch.uint8))


def _want_codes(p, out_scale):
    y, _ = oracle.gemm_reference(**dict(p.oracle_args(), c_dtype=wl.F32,
                                        C=np.zeros(p.M * p.ldc, np.int32)))
    t = torch.from_numpy(np.ascontiguousarray(y / out_scale)).to(torch.float32).clamp(-448, 448)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy(), y


@pytest.mark.parametrize("variant", ["pair", "two_pair_stream_k", "pair_tiles"])
@pytest.mark.parametrize("layout", ["NN", "TT"])
@pytest.mark.parametrize("ab", [wl.F16, wl.BF16, wl.E4M3], ids=["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("out_scale", [1.0, 2.0])
def test_fp8_output_exact(cuda_lib, variant, layout, ab, out_scale):
    g = cuda_lib
    g.gemm_set_multicast({"pair": 1, "two_pair_stream_k": 2, "pair_tiles": 1}[variant])
    g.gemm_set_schedule({"pair": 0, "two_pair_stream_k": 2, "pair_tiles": 1}[variant])
    try:
        # stream-K needs enough k-blocks per cluster: a larger, deeper problem there
        M, N, K = (1024, 1024, 4096) if variant == "two_pair_stream_k" else (520, 272, 64)
        p = _fp8_problem(300 + ab, M, N, K, ab, layout=layout, epilogue=wl.EPI_BIAS, ldc_pad=16)
        out, amax = run_ex(g, p, out_scale=out_scale)
        want, y = _want_codes(p, out_scale)
        got = out.reshape(p.M, p.ldc)[:, :p.N]
        assert np.array_equal(got, want.reshape(p.M, p.N))
        assert amax == float(np.abs(y).max())
    finally:
        g.gemm_set_multicast(g.MCAST_AUTO)
        g.gemm_set_schedule(g.SCHED_AUTO)


def test_fp8_output_simt_and_epilogue_only(cuda_lib):
    g = cuda_lib
    # misaligned A: the SIMT kernel
    p = _fp8_problem(310, 130, 72, 16, wl.BF16, epilogue=wl.EPI_BIAS_RELU)
    out, amax = run_ex(g, p, out_scale=0.5, a_offset=1)
    want, y = _want_codes(p, 0.5)
    assert np.array_equal(out.reshape(p.M, p.ldc)[:, :p.N], want.reshape(p.M, p.N))
    assert amax == float(np.abs(y).max())
    # alpha == 0: the epilogue-only kernel, y = bias
    p = _fp8_problem(311, 40, 72, 16, wl.F16, alpha=0.0, epilogue=wl.EPI_BIAS)
    out, amax = run_ex(g, p, out_scale=1.0)
    want, y = _want_codes(p, 1.0)
    assert np.array_equal(out.reshape(p.M, p.ldc)[:, :p.N], want.reshape(p.M, p.N))
    assert amax == float(np.abs(y).max())


@pytest.mark.parametrize("epi", [wl.EPI_NONE, wl.EPI_BIAS_GELU], ids=["none", "gelu"])
def test_fp8_workload_scaled_by_its_amax(cuda_lib, epi):
    """fp8 E4M3 inputs (per-tensor quantised) -> fp8 output quantised with the
    output's own amax: a first call measures amax, the second stores y / (amax/448)."""
    g = cuda_lib
    base = wl.fp8_e4m3(1024, c_dtype=wl.BF16)
    p = wl.dataclasses.replace(base, c_dtype=wl.E4M3, C=torch.zeros(base.M * base.ldc, dtype=torch.uint8),
                               epilogue=epi, bias=None if epi == wl.EPI_NONE else torch.full((base.N,), 0.1))
    _, amax = run_ex(g, p, out_scale=1.0)
    ref_amax, dmax = oracle.amax_reference(dict(p.oracle_args(), c_dtype=wl.F32, C=np.zeros(1, np.int32)))
    assert abs(amax - ref_amax) <= oracle.TOL_F32_OUT * dmax
    s = float(np.float32(amax / 448.0))
    out, _ = run_ex(g, p, out_scale=s, amax=False)
    res = oracle.check_fp8_output(p.oracle_args(), out, s)
    assert res["pass"], res


@pytest.mark.parametrize("case", ["bf16_out_transposable", "f16_out_stream_k", "fp32_3xtf32", "fp32_simt"])
def test_amax_with_other_outputs(cuda_lib, case):
    """amax alongside 16-bit and fp32 outputs; the outputs themselves stay within tolerance."""
    g = cuda_lib
    if case == "bf16_out_transposable":
        p = wl.random_problem(320, 640, 512, 256, wl.BF16, wl.BF16, layout="NN", epilogue=wl.EPI_BIAS_SILU)
        kw = {}
    elif case == "f16_out_stream_k":
        g.gemm_set_schedule(g.SCHED_STREAM_K)
        p = wl.random_problem(321, 1024, 1024, 512, wl.F16, wl.F16, alpha=1.5, beta=0.5)
        kw = {}
    elif case == "fp32_3xtf32":
        p = wl.random_problem(322, 200, 136, 96, wl.F32, wl.F32, alpha=2.0, beta=0.5)
        kw = {}
    else:
        p = wl.random_problem(323, 200, 136, 96, wl.F32, wl.F32, alpha=2.0, beta=0.5)
        kw = dict(use_workspace=False)
    try:
        out, amax = run_ex(g, p, **kw)
    finally:
        g.gemm_set_schedule(g.SCHED_AUTO)
    res = oracle.check(p.oracle_args(), out)
    assert res["pass"], res
    ref_amax, dmax = oracle.amax_reference(p.oracle_args())
    assert abs(amax - ref_amax) <= oracle.TOL_F32_OUT * dmax, (amax, ref_amax)


def test_fp8_output_rejections(cuda_lib):
    g = cuda_lib
    A = torch.zeros(64 * 64, dtype=torch.float16, device="cuda")
    C = torch.zeros(64 * 64, dtype=torch.uint8, device="cuda")
    for kw, ab in ((dict(beta=0.5), wl.F16), (dict(beta=0.0), wl.F32)):
        with pytest.raises(g.GemmError) as e:
            g.gemm_ex(64, 64, 64, ab, A, 64, 1, A, 64, 1, C, 64, wl.E4M3, 1.0, kw["beta"], None, wl.EPI_NONE)
        assert e.value.status == g.ERR_UNSUPPORTED
    with pytest.raises(g.GemmError) as e:      # gemm() itself has no fp8 output
        g.gemm(64, 64, 64, wl.F16, A, 64, 1, A, 64, 1, C, 64, wl.E4M3, 1.0, 0.0, None, wl.EPI_NONE)
    assert e.value.status == g.ERR_UNSUPPORTED
