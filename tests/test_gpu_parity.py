"""GPU parity: the CUDA library through its C ABI against the float64 oracle.

Bar: integer-valued inputs (exact in every storage type, sums < 2^24) must come
back bit-exact with fp32 output; random workloads must meet the normalised
tolerance (2e-3 for 16-bit outputs, 1e-5 for fp32 outputs).  Every run also
checks that nothing outside the M x N block of C was written (guards and ldc
padding compared bit for bit).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import run_gemm, sample_rows

pytestmark = pytest.mark.gpu

TC_SHAPES = [
    (128, 256, 128),     # one tile, two k-blocks (16-bit)
    (16, 16, 16),        # far smaller than a tile: TMA zero fill everywhere
    (336, 208, 1008),    # ragged M, N and K, 16-byte row pitches
    (256, 512, 1024),    # several tiles, ring wraps
    (2048, 2048, 256),   # several tiles per CTA: double-buffered accumulator
    (1024, 768, 4096),   # long K
]


def _assert_exact(run):
    y, _ = oracle.gemm_reference(**run.p.oracle_args())
    got = run.values()
    bad = np.argwhere(got != y)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:3].tolist()}: got {got[tuple(bad[0])]} " \
                          f"want {y[tuple(bad[0])]}"


# (policy, pair width): every tile variant of the tcgen05 path
POLICIES = [(1, 0), (2, 0), (3, 0), (3, 224), (3, 160)]


@pytest.fixture
def tile_policy(cuda_lib, request):
    policy, bn = request.param
    cuda_lib.gemm_set_tile_policy(policy, bn)
    yield request.param
    cuda_lib.gemm_set_tile_policy(cuda_lib.TILE_AUTO, 0)


@pytest.mark.parametrize("tile_policy", POLICIES, indirect=True, ids=lambda p: f"pol{p[0]}-{p[1]}")
@pytest.mark.parametrize("shape", TC_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("ab", [wl.F16, wl.BF16, wl.E4M3], ids=["f16", "bf16", "e4m3"])
def test_integer_exact_tcgen05(cuda_lib, ab, layout, shape, tile_policy):
    M, N, K = shape
    p = wl.random_problem(1000 + M + N + K, M, N, K, ab, wl.F32, layout=layout, alpha=2.0, beta=-1.0,
                          integer=True)
    r = run_gemm(cuda_lib, p)
    assert r.status == 0
    assert r.path == cuda_lib.PATH_TCGEN05
    _assert_exact(r)


@pytest.mark.parametrize("ab", [wl.F16, wl.BF16, wl.E4M3], ids=["f16", "bf16", "e4m3"])
def test_integer_exact_simt_fallback(cuda_lib, ab):
    """Row pitches that TMA cannot take run on the SIMT kernel, still exact."""
    for (M, N, K, layout) in [(5, 260, 129, "NN"), (77, 33, 301, "TT"), (130, 129, 67, "NT")]:
        p = wl.random_problem(7 + M, M, N, K, ab, wl.F32, layout=layout, alpha=1.0, beta=0.0, integer=True)
        r = run_gemm(cuda_lib, p)
        assert r.path == cuda_lib.PATH_SIMT
        _assert_exact(r)


def test_integer_exact_misaligned_base(cuda_lib):
    p = wl.random_problem(3, 256, 256, 256, wl.BF16, wl.F32, integer=True)
    r = run_gemm(cuda_lib, p, a_elem_offset=1)
    assert r.path == cuda_lib.PATH_SIMT
    _assert_exact(r)


@pytest.mark.parametrize("tile_policy", [(1, 0), (3, 0), (3, 192)], indirect=True, ids=lambda p: f"pol{p[0]}-{p[1]}")
@pytest.mark.parametrize("out", [wl.F16, wl.BF16, wl.F32], ids=["f16", "bf16", "f32"])
@pytest.mark.parametrize("epi", [wl.EPI_NONE, wl.EPI_BIAS, wl.EPI_BIAS_GELU], ids=["none", "bias", "gelu"])
def test_epilogues_and_outputs_ragged(cuda_lib, out, epi, tile_policy):
    for ab in (wl.F16, wl.BF16):
        p = wl.random_problem(31, 300, 200, 520, ab, out, alpha=0.75, beta=0.5 if epi == 0 else 0.0,
                              epilogue=epi)
        r = run_gemm(cuda_lib, p)
        assert r.path == cuda_lib.PATH_TCGEN05
        res = r.check()
        assert res["pass"], res


def test_odd_ldc_uses_masked_store(cuda_lib):
    p = wl.random_problem(41, 256, 256, 256, wl.BF16, wl.BF16, beta=1.0, ldc_pad=3, epilogue=wl.EPI_BIAS)
    r = run_gemm(cuda_lib, p)
    assert r.path == cuda_lib.PATH_TCGEN05 and r.check()["pass"]


# ------------------------------------------------------------------ workloads --

def test_fp32_256(cuda_lib):
    """fp32 with a workspace runs as 3xTF32 on the tensor cores (what the launch record says);
    gemm_query_path reports the path without one (the FFMA kernel), as the header documents."""
    r = run_gemm(cuda_lib, wl.fp32_square(256))
    assert r.path == cuda_lib.PATH_SIMT
    info = cuda_lib.gemm_last_launch()
    assert info["path"] == cuda_lib.PATH_TCGEN05 and info["tf32x3"] == 1
    res = r.check()
    assert res["pass"], res
    r = run_gemm(cuda_lib, wl.fp32_square(256), use_workspace=False)
    assert cuda_lib.gemm_last_launch()["path"] == cuda_lib.PATH_SIMT
    res = r.check()
    assert res["pass"], res


@pytest.mark.parametrize("n", [512, 1024, 2048, 1000])
def test_fp16_alpha_beta_full(cuda_lib, n):
    r = run_gemm(cuda_lib, wl.fp16_alpha_beta(n))
    assert r.path == cuda_lib.PATH_TCGEN05
    res = r.check()
    assert res["pass"], res


def test_fp16_alpha_beta_4096_sampled(cuda_lib):
    r = run_gemm(cuda_lib, wl.fp16_alpha_beta(4096))
    res = r.check(rows=sample_rows(4096))
    assert res["pass"], res


@pytest.mark.parametrize("M", [512, 2048])
def test_bias_gelu_fused_and_unfused(cuda_lib, M):
    g = cuda_lib
    p = wl.bf16_bias_gelu(M)
    r = run_gemm(g, p)
    assert r.path == g.PATH_TCGEN05
    res = r.check()
    assert res["pass"], res
    # decomposed path: GEMM with no epilogue, then the separate bias+GELU pass
    A, B, bias = p.A.cuda(), p.B.cuda(), p.bias.cuda()
    C = torch.empty(p.M * p.ldc, dtype=torch.bfloat16, device="cuda")
    g.gemm(p.M, p.N, p.K, p.ab_dtype, A, p.a_stride_m, p.a_stride_k, B, p.b_stride_k, p.b_stride_n, C, p.ldc,
           p.c_dtype, p.alpha, 0.0, None, wl.EPI_NONE)
    g.gemm_bias_gelu(p.M, p.N, C, p.ldc, p.c_dtype, bias)
    assert g.gemm_device_status() == 0
    out = C.cpu().view(torch.int16).numpy()
    res2 = oracle.check(p.oracle_args(), out)
    assert res2["pass"], res2


def test_bias_gelu_8192_sampled(cuda_lib):
    r = run_gemm(cuda_lib, wl.bf16_bias_gelu(8192))
    res = r.check(rows=sample_rows(8192))
    assert res["pass"], res


def test_fp8_2048_full_bf16_and_f32_out(cuda_lib):
    r = run_gemm(cuda_lib, wl.fp8_e4m3(2048))
    assert r.path == cuda_lib.PATH_TCGEN05
    res = r.check()
    assert res["pass"], res
    r32 = run_gemm(cuda_lib, wl.fp8_e4m3(2048, c_dtype=wl.F32))
    res32 = r32.check()
    assert res32["pass"], res32


@pytest.mark.parametrize("n", [4096, 8192])
def test_fp8_sampled(cuda_lib, n):
    r = run_gemm(cuda_lib, wl.fp8_e4m3(n))
    res = r.check(rows=sample_rows(n))
    assert res["pass"], res


@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
def test_fp32_layouts_4096_sampled(cuda_lib, layout):
    r = run_gemm(cuda_lib, wl.fp32_layout(layout, 4096))
    res = r.check(rows=sample_rows(4096, n_random=64))
    assert res["pass"], res


def test_bf16_nn_8192_sampled(cuda_lib):
    r = run_gemm(cuda_lib, wl.bf16_nn_large(8192))
    assert r.path == cuda_lib.PATH_TCGEN05
    res = r.check(rows=sample_rows(8192, n_random=128))
    assert res["pass"], res


# ------------------------------------------------------------- degenerate cases --

def test_m_or_n_zero_is_noop(cuda_lib):
    g = cuda_lib
    C = torch.full((64,), 7.0, device="cuda")
    g.gemm(0, 8, 8, g.F32, None, 8, 1, None, 8, 1, C, 8, g.F32, 1.0, 1.0, None, 0)
    g.gemm(8, 0, 8, g.F32, None, 8, 1, None, 8, 1, C, 8, g.F32, 1.0, 1.0, None, 0)
    assert g.gemm_device_status() == 0
    assert bool((C == 7.0).all())


@pytest.mark.parametrize("out", [wl.F16, wl.F32], ids=["f16", "f32"])
@pytest.mark.parametrize("kind", ["k0", "alpha0"])
def test_epilogue_only(cuda_lib, kind, out):
    # Here |z| is of the order of the error scale D itself, so a bf16 output's
    # rounding (unit roundoff 2^-8) alone would exceed 2e-3: f16 / f32 outputs.
    K = 0 if kind == "k0" else 64
    alpha = 1.0 if kind == "k0" else 0.0
    p = wl.random_problem(51, 130, 70, K, wl.BF16, out, alpha=alpha, beta=0.5, epilogue=wl.EPI_BIAS_GELU)
    r = run_gemm(cuda_lib, p)
    assert r.path == cuda_lib.PATH_EPILOGUE_ONLY
    res = r.check()
    assert res["pass"], res


@pytest.mark.parametrize("ab,out", [(wl.BF16, wl.BF16), (wl.F32, wl.F32), (wl.E4M3, wl.F32)])
def test_beta_zero_never_reads_c(cuda_lib, ab, out):
    p = wl.random_problem(61, 200, 136, 96, ab, out, alpha=1.0, beta=0.0)
    r = run_gemm(cuda_lib, p, nan_c=True)
    assert not np.isnan(r.values()).any()
    assert r.check()["pass"]


def test_runs_on_a_side_stream(cuda_lib):
    s = torch.cuda.Stream()
    p = wl.fp16_alpha_beta(384, 256, 320)
    with torch.cuda.stream(s):
        r = run_gemm(cuda_lib, p, stream=s)
    assert r.check()["pass"]


def test_deterministic(cuda_lib):
    p = wl.bf16_bias_gelu(512, N=1024, K=1024)
    a = run_gemm(cuda_lib, p).out_codes
    b = run_gemm(cuda_lib, p).out_codes
    assert np.array_equal(a, b)


def test_bounded_waits_give_up_and_report(cuda_lib):
    """A wait that can never complete ends after its limit with a timeout status;
    the context stays usable and the status clears once read."""
    import time
    g = cuda_lib
    assert g.gemm_device_status() == g.OK
    flag = torch.zeros(4, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    g.gemm_wait_selftest(flag, 20_000_000)  # 20 ms per wait
    assert g.gemm_device_status() == g.ERR_TIMEOUT
    assert 0.03 < time.perf_counter() - t0 < 5.0
    assert g.gemm_device_status() == g.OK
    r = run_gemm(g, wl.random_problem(5, 256, 256, 256, wl.BF16, wl.F32, integer=True))
    _assert_exact(r)
    with pytest.raises(g.GemmError):
        g.gemm_wait_selftest(flag, 2_000_000_000)


def test_rejects_pageable_host_and_out_of_range_buffers(cuda_lib):
    g = cuda_lib
    A = torch.zeros(64 * 64, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(64 * 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(64 * 64, dtype=torch.bfloat16, device="cuda")
    host = torch.zeros(64 * 64, dtype=torch.bfloat16)
    with pytest.raises(g.GemmError) as ei:
        g.gemm(64, 64, 64, g.BF16, host, 64, 1, B, 64, 1, C, 64, g.BF16, 1.0, 0.0, None, 0)
    assert ei.value.status == g.ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as ei:
        g.gemm(64, 64, 64, g.BF16, A, 1 << 34, 1, B, 64, 1, C, 64, g.BF16, 1.0, 0.0, None, 0)
    assert ei.value.status == g.ERR_INVALID_ARG
    assert g.gemm_device_status() == 0


def test_cost_model_choices(cuda_lib):
    g = cuda_lib
    g.gemm_set_tile_policy(g.TILE_AUTO, 0)
    kind, bn, units = g.gemm_query_tile(4096, 4096, 4096, g.F16, g.F16)
    assert kind == 2 and bn == 256 and units >= 70   # pair of SMs
    kind, bn, _ = g.gemm_query_tile(8192, 8192, 8192, g.BF16, g.BF16)
    assert kind == 2 and bn == 256
    g.gemm_set_tile_policy(g.TILE_1SM_128, 0)
    assert g.gemm_query_tile(4096, 4096, 4096, g.F16, g.F16)[:2] == (1, 128)
    g.gemm_set_tile_policy(g.TILE_PAIR, 160)
    assert g.gemm_query_tile(4096, 4096, 4096, g.F16, g.F16)[:2] == (2, 160)
    g.gemm_set_tile_policy(g.TILE_AUTO, 0)


@pytest.mark.parametrize("tile_policy", [(1, 0), (3, 256), (3, 224)], indirect=True, ids=lambda p: f"pol{p[0]}-{p[1]}")
def test_fp16_alpha_beta_2048_each_tiling(cuda_lib, tile_policy):
    r = run_gemm(cuda_lib, wl.fp16_alpha_beta(2048))
    res = r.check()
    assert res["pass"], res
    assert cuda_lib.gemm_device_status() == 0


@pytest.mark.parametrize("ab", [wl.BF16, wl.F32], ids=["tcgen05", "simt"])
def test_gelu_accuracy_over_range(cuda_lib, ab):
    """z = bias exactly (the product is zero); fp32 output against float64 GELU."""
    g = cuda_lib
    M, N, K = 128, 4096, 64
    a = torch.zeros(M, K)
    b = torch.zeros(K, N)
    bias = torch.linspace(-9.0, 9.0, N, dtype=torch.float32)
    p = wl.make_problem("gelu_range", M, N, K, ab, wl.F32, a, b, alpha=1.0, beta=0.0, bias=bias,
                        epilogue=wl.EPI_BIAS_GELU)
    r = run_gemm(g, p)
    assert r.path == (g.PATH_TCGEN05 if ab == wl.BF16 else g.PATH_SIMT)
    got = r.values()
    z = bias.double().numpy()
    want = oracle.gelu(z)[None, :]
    err = np.abs(got - want)
    assert float(err.max()) <= 2e-7 * 9, float(err.max())
    assert np.all(err <= 1e-7 + 4e-7 * np.abs(z)[None, :])
    # and the stated metric itself: normalised error with D = |z| (times max|GELU'|) within 1e-5
    D = np.broadcast_to(np.abs(z)[None, :], got.shape)
    assert oracle.max_normalized_error(got, want, D, wl.EPI_BIAS_GELU) <= 1e-5


# ---------------------------------------------------------------- stream-K --

@pytest.fixture
def schedule(cuda_lib, request):
    cuda_lib.gemm_set_schedule(request.param)
    yield request.param
    cuda_lib.gemm_set_schedule(cuda_lib.SCHED_AUTO)


SK_SHAPES = [(256, 256, 1024), (512, 768, 4096), (336, 208, 3008), (1024, 1024, 2048), (128, 4096, 1024)]


@pytest.mark.parametrize("schedule", [2], indirect=True, ids=["streamk"])
@pytest.mark.parametrize("shape", SK_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout", ["NN", "TT"])
@pytest.mark.parametrize("ab", [wl.BF16, wl.E4M3], ids=["bf16", "e4m3"])
def test_integer_exact_stream_k(cuda_lib, ab, layout, shape, schedule):
    """Every tile's k-blocks split over all SM pairs: partial sums through the
    workspace must reproduce the exact integer result (sums < 2^24)."""
    M, N, K = shape
    p = wl.random_problem(500 + M + K, M, N, K, ab, wl.F32, layout=layout, alpha=2.0, beta=-1.0,
                          integer=True)
    r = run_gemm(cuda_lib, p)
    assert r.status == 0 and r.path == cuda_lib.PATH_TCGEN05
    _assert_exact(r)


@pytest.mark.parametrize("schedule", [0, 1, 2], indirect=True, ids=["auto", "tiles", "streamk"])
@pytest.mark.parametrize("epi", [wl.EPI_NONE, wl.EPI_BIAS_GELU], ids=["none", "gelu"])
def test_schedules_agree(cuda_lib, epi, schedule):
    """Random data, every schedule within tolerance; whole-tile vs stream-K sums
    differ only in the order of fp32 additions."""
    p = wl.random_problem(77, 1536, 1280, 2048, wl.BF16, wl.F32, alpha=0.5, beta=0.0, epilogue=epi)
    r = run_gemm(cuda_lib, p)
    res = r.check()
    assert res["pass"], res


def test_stream_k_repeated_calls_and_no_workspace(cuda_lib):
    """Flags reset after use: back-to-back stream-K calls on one workspace stay
    correct, and a call without workspace falls back to whole tiles."""
    g = cuda_lib
    g.gemm_set_schedule(g.SCHED_STREAM_K)
    try:
        p = wl.random_problem(88, 640, 512, 1536, wl.F16, wl.F32, alpha=1.0, beta=1.0, integer=True)
        for _ in range(3):
            _assert_exact(run_gemm(g, p))
        _assert_exact(run_gemm(g, p, use_workspace=False))
    finally:
        g.gemm_set_schedule(g.SCHED_AUTO)


def test_workspace_size(cuda_lib):
    g = cuda_lib
    n = g.gemm_workspace_size(4096, 4096, 4096, g.F16)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert n >= (sms // 2) * 2 * 128 * 256 * 4
    # fp32 inputs: the 3xTF32 split of A and B (hi + lo, K-major, 16-byte rows)
    assert g.gemm_workspace_size(4096, 4096, 4096, g.F32) == 2 * (4096 + 4096) * 4096 * 4
    assert g.gemm_workspace_size(100, 50, 9, g.F32) == 256 * ((2 * 100 * 12 * 4 + 255) // 256) + 256 * (
        (2 * 50 * 12 * 4 + 255) // 256)


# ------------------------------------------------------------------- 3xTF32 --

@pytest.mark.parametrize("shape", [(256, 256, 128), (336, 200, 1000), (1024, 768, 4096), (5, 300, 77)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
def test_fp32_3xtf32_integer_exact(cuda_lib, layout, shape):
    """Small integers are exact in tf32 (lo = 0): the split path must be exact."""
    M, N, K = shape
    p = wl.random_problem(900 + M + K, M, N, K, wl.F32, wl.F32, layout=layout, alpha=2.0, beta=-1.0,
                          integer=True, ldc_pad=3)
    r = run_gemm(cuda_lib, p)
    assert r.status == 0
    _assert_exact(r)


def test_fp32_workspace_selects_tensor_core_path(cuda_lib):
    """With a workspace fp32 runs as 3xTF32 (tensor cores), without it on the FFMA
    kernel; both meet 1e-5 and their roundings differ."""
    p = wl.random_problem(123, 768, 640, 2048, wl.F32, wl.F32, alpha=1.0, beta=0.5)
    a = run_gemm(cuda_lib, p, use_workspace=True)
    b = run_gemm(cuda_lib, p, use_workspace=False)
    ra, rb = a.check(), b.check()
    assert ra["pass"] and rb["pass"], (ra, rb)
    assert not np.array_equal(a.out_codes, b.out_codes)
