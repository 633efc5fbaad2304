"""GPU parity of the pair kernel's two-pair clusters (A shared by TMA multicast).

Two SM pairs of one cluster compute two tiles side by side along N; each CTA
fetches half of its A rows and the TMA delivers them to both pairs.  Only the
data movement changes, so the bar is the one of the one-pair kernel:

* integer-valued inputs (sums < 2^24, exact in fp32 accumulation) come back
  bit-exact against the float64 oracle, in every layout, ragged shape, tile
  width and schedule, including a forced odd number of tile columns (the last
  pair then computes a tile outside the matrix and must store nothing);
* random workloads meet the normalised tolerance, and with whole tiles the
  output is bit-identical to the one-pair kernel's (same MMAs in the same
  order on the same operands).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import run_gemm

pytestmark = pytest.mark.gpu

SHAPES = [
    (128, 256, 128),     # one tile column: the second pair lies outside the matrix
    (16, 16, 16),        # far smaller than a tile
    (336, 208, 1008),    # ragged M, N, K
    (256, 1024, 1024),   # two tile pairs side by side
    (2048, 2048, 256),   # several tile pairs per cluster
    (1024, 768, 4096),   # long K, odd number of tile columns
]


@pytest.fixture
def mcast_on(cuda_lib):
    cuda_lib.gemm_set_multicast(cuda_lib.MCAST_ON)
    cuda_lib.gemm_set_tile_policy(cuda_lib.TILE_PAIR, 0)
    yield
    cuda_lib.gemm_set_multicast(cuda_lib.MCAST_AUTO)
    cuda_lib.gemm_set_tile_policy(cuda_lib.TILE_AUTO, 0)
    cuda_lib.gemm_set_schedule(cuda_lib.SCHED_AUTO)
    cuda_lib.gemm_set_operand_order(cuda_lib.ORDER_AUTO)


def _assert_exact(run):
    y, _ = oracle.gemm_reference(**run.p.oracle_args())
    got = run.values()
    bad = np.argwhere(got != y)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:3].tolist()}: got {got[tuple(bad[0])]} " \
                          f"want {y[tuple(bad[0])]}"


@pytest.mark.parametrize("sched", ["auto", "tiles", "stream_k"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("ab", [wl.F16, wl.BF16, wl.E4M3], ids=["f16", "bf16", "e4m3"])
def test_integer_exact_two_pair_clusters(cuda_lib, mcast_on, ab, layout, shape, sched):
    g = cuda_lib
    g.gemm_set_schedule({"auto": g.SCHED_AUTO, "tiles": g.SCHED_TILES, "stream_k": g.SCHED_STREAM_K}[sched])
    M, N, K = shape
    p = wl.random_problem(2000 + M + N + K, M, N, K, ab, wl.F32, layout=layout, alpha=2.0, beta=-1.0,
                          integer=True)
    r = run_gemm(g, p)
    assert r.status == 0
    assert r.path == g.PATH_TCGEN05
    _assert_exact(r)


@pytest.mark.parametrize("bn", [128, 160, 224])
def test_integer_exact_two_pair_clusters_widths(cuda_lib, mcast_on, bn):
    g = cuda_lib
    g.gemm_set_tile_policy(g.TILE_PAIR, bn)
    for ab, layout in ((wl.BF16, "NN"), (wl.F16, "TT"), (wl.E4M3, "NT")):
        p = wl.random_problem(77 + bn, 528, 1000, 640, ab, wl.F32, layout=layout, alpha=1.0, beta=0.5,
                              integer=True)
        r = run_gemm(g, p)
        assert r.status == 0
        _assert_exact(r)


@pytest.mark.parametrize("order", ["given", "transposed"])
def test_two_pair_clusters_transposed_order(cuda_lib, mcast_on, order):
    """C^T = B^T A^T with two pairs per cluster: 16-bit outputs rounded exactly."""
    g = cuda_lib
    g.gemm_set_operand_order(g.ORDER_AS_GIVEN if order == "given" else g.ORDER_TRANSPOSED)
    for layout in ("NN", "NT", "TN", "TT"):
        p = wl.random_problem(91, 528, 304, 272, wl.BF16, wl.BF16, layout=layout, alpha=1.0, beta=1.0,
                              integer=True)
        r = run_gemm(g, p)
        assert r.status == 0
        y, _ = oracle.gemm_reference(**p.oracle_args())
        want = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float32).to(torch.bfloat16)
        assert np.array_equal(r.values(), want.to(torch.float64).numpy())


def _output_codes(g, p, mcast):
    g.gemm_set_multicast(mcast)
    return run_gemm(g, p)


@pytest.mark.parametrize("epi", [wl.EPI_NONE, wl.EPI_BIAS_GELU], ids=["none", "gelu"])
def test_random_workloads_match_one_pair_kernel_bitwise(cuda_lib, mcast_on, epi):
    g = cuda_lib
    g.gemm_set_schedule(g.SCHED_TILES)
    if epi == wl.EPI_NONE:
        p = wl.fp16_alpha_beta(2048)
    else:
        p = wl.bf16_bias_gelu(2048)
    on = _output_codes(g, p, g.MCAST_ON)
    off = _output_codes(g, p, g.MCAST_OFF)
    assert on.status == 0 and off.status == 0
    res = on.check()
    assert res["pass"], res
    assert np.array_equal(on.out_codes, off.out_codes)


def test_fp16_headline_shape_stream_k_tolerance(cuda_lib, mcast_on):
    """fp16 4096^3 alpha/beta workload on two-pair clusters with the stream-K tail (sampled rows)."""
    from gpu_util import sample_rows
    g = cuda_lib
    g.gemm_set_multicast(g.MCAST_AUTO)
    g.gemm_set_tile_policy(g.TILE_AUTO, 0)
    g.gemm_set_schedule(g.SCHED_STREAM_K)
    r = run_gemm(g, wl.fp16_alpha_beta(4096))
    assert r.status == 0
    res = r.check(rows=sample_rows(4096))
    assert res["pass"], res


def test_launch_record_matches_the_chosen_shape(cuda_lib):
    """gemm_last_launch reports what ran: the transposed pair kernel at fp16 4096^3, with two-pair
    clusters under AUTO (4 waves of tiles or fewer, even tile columns), and the shape the knob forces."""
    g = cuda_lib
    p = wl.fp16_alpha_beta(4096)
    r = run_gemm(g, p)
    assert r.status == 0
    info = g.gemm_last_launch()
    assert info["path"] == g.PATH_TCGEN05 and info["kind"] == 2 and info["bn"] == 256
    # A row-major, B row-major fp16 with 16-bit output: the pair kernel runs C^T = B^T A^T
    assert info["transposed"] == 1
    assert info["cluster_ctas"] in (2, 4) and info["grid_ctas"] % info["cluster_ctas"] == 0
    assert info["tiles"] == (256 if info["cluster_ctas"] == 2 else 128)
    try:
        g.gemm_set_multicast(g.MCAST_OFF)
        run_gemm(g, p)
        off = g.gemm_last_launch()
        assert off["cluster_ctas"] == 2 and off["tiles"] == 256
        g.gemm_set_multicast(g.MCAST_ON)
        run_gemm(g, p)
        on = g.gemm_last_launch()
        assert on["cluster_ctas"] == 4 and on["tiles"] == 128
        # AUTO: two-pair clusters if they lose no SM pair or the problem has at most 4 waves of tiles
        if 2 * (on["grid_ctas"] // 4) >= off["grid_ctas"] // 2 or 256 <= 4 * (off["grid_ctas"] // 2):
            assert info["cluster_ctas"] == 4
    finally:
        g.gemm_set_multicast(g.MCAST_AUTO)


def test_launch_record_fp32_paths(cuda_lib):
    g = cuda_lib
    p = wl.fp32_square(256)
    run_gemm(g, p)
    info = g.gemm_last_launch()
    assert info["path"] == g.PATH_TCGEN05 and info["tf32x3"] == 1 and info["cluster_ctas"] == 2
    run_gemm(g, p, use_workspace=False)
    info = g.gemm_last_launch()
    assert info["path"] == g.PATH_SIMT and info["tf32x3"] == 0 and info["grid_ctas"] == 0


def _run_placed(g, p, pinned):
    """Run p with the operands named in `pinned` ("A", "B") in pinned host memory, the rest on the device."""
    A = p.A.pin_memory() if "A" in pinned else p.A.cuda()
    B = p.B.pin_memory() if "B" in pinned else p.B.cuda()
    C = p.C.clone().cuda()
    ws = torch.empty(g.gemm_workspace_size(p.M, p.N, p.K, p.ab_dtype), dtype=torch.uint8, device="cuda")
    g.gemm(p.M, p.N, p.K, p.ab_dtype, A, p.a_stride_m, p.a_stride_k, B, p.b_stride_k, p.b_stride_n, C, p.ldc,
           p.c_dtype, p.alpha, p.beta, None, p.epilogue, workspace=ws, workspace_bytes=ws.numel())
    info = g.gemm_last_launch()
    assert g.gemm_device_status() == 0
    torch.cuda.synchronize()
    return info, oracle.output_values(C.cpu().view(wl.CODE_VIEW[p.c_dtype]).numpy(), p.M, p.N, p.ldc, p.c_dtype)


@pytest.mark.parametrize("pinned, order, want_cl", [
    ("A", "given", 2),        # the multicast operand is host memory: one-pair clusters
    ("B", "given", 4),        # B is not multicast; A (device memory) may be
    ("B", "transposed", 2),   # C^T = B^T A^T: B is now the multicast operand
    ("", "given", 4),         # both on the device
])
def test_multicast_only_over_this_devices_memory(cuda_lib, mcast_on, pinned, order, want_cl):
    """A multicast tensor map covers only this GPU's own memory: when the pair kernel's first
    operand lives in pinned host memory the call runs one-pair clusters even under MCAST_ON, and
    the result is the same exact product."""
    g = cuda_lib
    g.gemm_set_operand_order(g.ORDER_AS_GIVEN if order == "given" else g.ORDER_TRANSPOSED)
    c_dtype = wl.F32 if order == "given" else wl.BF16  # the transposed order needs a 16-bit output
    p = wl.random_problem(431, 512, 1024, 320, wl.BF16, c_dtype, alpha=1.0, beta=0.0, integer=True)
    info, got = _run_placed(g, p, pinned)
    assert info["kind"] == 2 and info["transposed"] == (order == "transposed")
    assert info["cluster_ctas"] == want_cl
    y, _ = oracle.gemm_reference(**p.oracle_args())
    if c_dtype == wl.F32:
        assert np.array_equal(got, y)
    else:
        want = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float32).to(torch.bfloat16)
        assert np.array_equal(got, want.to(torch.float64).numpy())
