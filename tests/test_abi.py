"""The C-ABI library (CPU only: no kernel launches).

* the shared library loads and exports every function include/*.h declares;
* the host-side argument validation and kernel-family choice, which run
  before any CUDA call, behave as the header documents.
"""
import ctypes
import glob
import os
import re

import pytest

from conftest import REPO


@pytest.fixture(scope="module")
def g():
    import __graft_entry__
    __graft_entry__.build()
    import dense_gemm_epilogues_tcgen05_gb300 as g
    return g


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(REPO, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b([A-Za-z_]\w*)\s*\(([^;{}]*)\)\s*;", text):
            if m.group(1) not in ("if", "while", "for", "return", "sizeof"):
                names.add(m.group(1))
    return names


def test_header_declares_the_entry_points():
    names = _declared_functions()
    assert {"gemm", "gemm_workspace_size", "gemm_query_path", "gemm_bias_gelu", "gemm_device_status",
            "gemm_status_string", "gemm_version", "gemm_set_tile_policy", "gemm_query_tile",
            "gemm_set_schedule", "gemm_builtin_scratch", "gemm_wait_selftest", "gemm_set_multicast",
            "gemm_last_launch", "gemm_q4", "gemm_set_q4_kernel", "gemm_get_tuning"} <= names


def test_library_exports_every_declared_symbol(g):
    lib = ctypes.CDLL(g.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(g):
    assert g.gemm_status_string(0) == "ok"
    assert "timed out" in g.gemm_status_string(6)
    assert g.gemm_status_string(99) == "unknown status"
    assert "sm_103a" in g.gemm_version()


def test_workspace_size_without_gpu(g):
    # fp32: the 3xTF32 split buffers, a pure function of the sizes
    assert g.gemm_workspace_size(4096, 4096, 4096, g.F32) == 2 * (4096 + 4096) * 4096 * 4
    assert g.gemm_workspace_size(0, 4096, 4096, g.F32) == 0
    # 16-bit / fp8: stream-K scratch per SM pair; without a device it is unknown: 0
    assert g.gemm_workspace_size(4096, 4096, 4096, g.BF16) >= 0


def test_schedule_validation(g):
    for v in (0, 1, 2):
        assert g.gemm_set_schedule(v) == 0
    for v in (-1, 3):
        with pytest.raises(g.GemmError):
            g.gemm_set_schedule(v)
    g.gemm_set_schedule(g.SCHED_AUTO)


def test_operand_order_validation(g):
    for v in (g.ORDER_AUTO, g.ORDER_AS_GIVEN, g.ORDER_TRANSPOSED):
        assert g.gemm_set_operand_order(v) == 0
    for v in (-1, 3):
        with pytest.raises(g.GemmError):
            g.gemm_set_operand_order(v)
    g.gemm_set_operand_order(g.ORDER_AUTO)


def test_q4_kernel_validation(g):
    for v in (g.Q4_AUTO, g.Q4_FFMA, g.Q4_MMA):
        assert g.gemm_set_q4_kernel(v) == 0
    for v in (-1, 3):
        with pytest.raises(g.GemmError):
            g.gemm_set_q4_kernel(v)
    g.gemm_set_q4_kernel(g.Q4_AUTO)


def test_last_launch_records_only_successful_calls(g):
    """A no-op call (M = 0) is recorded without touching a device; a rejected call is not."""
    assert g.gemm(0, 16, 16, g.F16, 0, 16, 1, 0, 16, 1, 0, 16, g.F16, 1.0, 0.0, None, g.EPI_NONE, stream=0) == 0
    info = g.gemm_last_launch()
    assert info["path"] == g.PATH_NOOP and info["grid_ctas"] == 0 and info["kind"] == 0
    with pytest.raises(g.GemmError):
        g.gemm(-1, 16, 16, g.F16, 0, 16, 1, 0, 16, 1, 0, 16, g.F16, 1.0, 0.0, None, g.EPI_NONE, stream=0)
    assert g.gemm_last_launch() == info
    assert set(info) == {"path", "kind", "bn", "transposed", "cluster_ctas", "grid_ctas", "tiles",
                         "stream_k_tiles", "tf32x3"}


def test_multicast_validation(g):
    for v in (g.MCAST_AUTO, g.MCAST_OFF, g.MCAST_ON):
        assert g.gemm_set_multicast(v) == 0
    for v in (-1, 3):
        with pytest.raises(g.GemmError):
            g.gemm_set_multicast(v)
    g.gemm_set_multicast(g.MCAST_AUTO)


def test_tuning_settings_are_per_thread(g):
    """A setting made in one thread leaves every other thread on AUTO (its own defaults)."""
    import threading
    auto = {"tile_policy": g.TILE_AUTO, "tile_bn": 0, "schedule": g.SCHED_AUTO, "operand_order": g.ORDER_AUTO,
            "multicast": g.MCAST_AUTO, "q4_kernel": g.Q4_AUTO}
    assert g.gemm_get_tuning() == auto
    seen = {}
    ready, release = threading.Event(), threading.Event()

    def tuner():
        g.gemm_set_tile_policy(g.TILE_PAIR, 192)
        g.gemm_set_schedule(g.SCHED_STREAM_K)
        g.gemm_set_operand_order(g.ORDER_TRANSPOSED)
        g.gemm_set_multicast(g.MCAST_OFF)
        g.gemm_set_q4_kernel(g.Q4_MMA)
        seen["tuner"] = g.gemm_get_tuning()
        ready.set()
        release.wait(10)

    def other():
        ready.wait(10)
        seen["other"] = g.gemm_get_tuning()

    t1, t2 = threading.Thread(target=tuner), threading.Thread(target=other)
    t1.start(); t2.start()
    t2.join(10)
    release.set()
    t1.join(10)
    assert seen["tuner"] == {"tile_policy": g.TILE_PAIR, "tile_bn": 192, "schedule": g.SCHED_STREAM_K,
                             "operand_order": g.ORDER_TRANSPOSED, "multicast": g.MCAST_OFF, "q4_kernel": g.Q4_MMA}
    assert seen["other"] == auto
    assert g.gemm_get_tuning() == auto  # this thread too


# Fake, aligned device addresses: query_path never dereferences them.
PA, PB, PC, PBIAS = 0x7F0000000000, 0x7F1000000000, 0x7F2000000000, 0x7F3000000000


def q(g, M=256, N=256, K=256, ab=None, A=PA, sam=256, sak=1, B=PB, sbk=256, sbn=1, C=PC, ldc=256, cd=None,
      alpha=1.0, beta=0.0, bias=None, epi=0):
    ab = g.BF16 if ab is None else ab
    cd = g.BF16 if cd is None else cd
    return g.gemm_query_path(M, N, K, ab, A, sam, sak, B, sbk, sbn, C, ldc, cd, alpha, beta, bias, epi)


def test_path_choice_by_layout(g):
    # NN (A K-major, B N-major), NT, TN, TT: all on the tensor cores
    assert q(g) == g.PATH_TCGEN05
    assert q(g, sbk=1, sbn=256) == g.PATH_TCGEN05
    assert q(g, sam=1, sak=256) == g.PATH_TCGEN05
    assert q(g, sam=1, sak=256, sbk=1, sbn=256) == g.PATH_TCGEN05
    assert q(g, ab=g.E4M3) == g.PATH_TCGEN05
    assert q(g, ab=g.F16, cd=g.F32) == g.PATH_TCGEN05


def test_path_choice_fallbacks(g):
    assert q(g, ab=g.F32, cd=g.F32) == g.PATH_SIMT                    # fp32 inputs: FFMA kernel
    assert q(g, A=PA + 2) == g.PATH_SIMT                               # base not 16-byte aligned
    assert q(g, K=1001, sam=1001) == g.PATH_SIMT                       # row pitch not a multiple of 16 B
    assert q(g, K=1000, sam=1000) == g.PATH_TCGEN05                    # 2000 B pitch is fine
    assert q(g, sam=512, sak=2) == g.PATH_SIMT                         # no unit stride
    assert q(g, M=1, sam=3) == g.PATH_TCGEN05                          # single row: pitch unused
    assert q(g, ab=g.E4M3, K=24, sam=24) == g.PATH_SIMT                # 24 B pitch


def test_degenerate_paths(g):
    assert q(g, M=0) == g.PATH_NOOP
    assert q(g, N=0, A=None, B=None, C=None) == g.PATH_NOOP
    assert q(g, K=0, A=None, B=None) == g.PATH_EPILOGUE_ONLY
    assert q(g, alpha=0.0, A=None, B=None) == g.PATH_EPILOGUE_ONLY


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1), 1), (dict(K=-5), 1), (dict(ldc=255), 1), (dict(C=None), 1), (dict(A=None), 1),
    (dict(epi=1), 1), (dict(epi=6, bias=PBIAS), 1), (dict(epi=-1, bias=PBIAS), 1), (dict(ab=7), 1), (dict(sam=-256), 1),
    (dict(ab=0, cd=2), 2), (dict(ab=3, cd=1), 2), (dict(cd=3), 2), (dict(M=1 << 31), 2),
])
def test_argument_errors(g, kw, status):
    with pytest.raises(g.GemmError) as ei:
        q(g, **kw)
    assert ei.value.status == status


def test_gemm_rejects_bad_arguments_before_any_cuda_call(g):
    with pytest.raises(g.GemmError) as ei:
        g.gemm(-1, 4, 4, g.BF16, PA, 4, 1, PB, 4, 1, PC, 4, g.BF16, 1.0, 0.0, None, 0, stream=0)
    assert ei.value.status == g.ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as ei:
        g.gemm(4, 4, 4, g.F32, PA, 4, 1, PB, 4, 1, PC, 4, g.F16, 1.0, 0.0, None, 0, stream=0)
    assert ei.value.status == g.ERR_UNSUPPORTED
    # M == 0: a no-op that succeeds without touching anything
    assert g.gemm(0, 4, 4, g.BF16, None, 4, 1, None, 4, 1, None, 4, g.BF16, 1.0, 0.0, None, 0, stream=0) == 0


def test_tile_policy_validation(g):
    for policy, bn in [(0, 0), (1, 0), (2, 0), (3, 0), (3, 128), (3, 224), (3, 256)]:
        assert g.gemm_set_tile_policy(policy, bn) == 0
    for policy, bn in [(4, 0), (-1, 0), (3, 96), (3, 288), (3, 200), (1, 256)]:
        with pytest.raises(g.GemmError) as ei:
            g.gemm_set_tile_policy(policy, bn)
        assert ei.value.status == g.ERR_INVALID_ARG
    g.gemm_set_tile_policy(g.TILE_AUTO, 0)


def test_baseline_validation_without_gpu(g):
    """Argument and support checks of gemm_baseline happen on the host, before any CUDA call."""
    A, B, C = 0x100000, 0x200000, 0x300000  # 16-byte aligned stand-ins, never dereferenced
    with pytest.raises(g.GemmError) as e:
        g.gemm_baseline(7, 64, 64, 64, g.F16, A, 64, 1, B, 64, 1, C, 64, g.F16, 1.0, 0.0, None, g.EPI_NONE,
                        stream=0)
    assert e.value.status == g.ERR_INVALID_ARG
    # mma.sync: fp16 / bf16 only
    with pytest.raises(g.GemmError) as e:
        g.gemm_baseline(g.BASELINE_MMA_SYNC, 64, 64, 64, g.F32, A, 64, 1, B, 64, 1, C, 64, g.F32, 1.0, 0.0, None,
                        g.EPI_NONE, stream=0)
    assert e.value.status == g.ERR_UNSUPPORTED
    # mma.sync: K-contiguous A needs K % 8 == 0
    with pytest.raises(g.GemmError) as e:
        g.gemm_baseline(g.BASELINE_MMA_SYNC, 64, 64, 60, g.F16, A, 64, 1, B, 64, 1, C, 64, g.F16, 1.0, 0.0, None,
                        g.EPI_NONE, stream=0)
    assert e.value.status == g.ERR_UNSUPPORTED
    # mma.sync: strides the TMA could not take (odd row pitch)
    with pytest.raises(g.GemmError) as e:
        g.gemm_baseline(g.BASELINE_MMA_SYNC, 64, 64, 64, g.F16, A, 65, 1, B, 64, 1, C, 64, g.F16, 1.0, 0.0, None,
                        g.EPI_NONE, stream=0)
    assert e.value.status == g.ERR_UNSUPPORTED
    # no-op sizes succeed without a device
    assert g.gemm_baseline(g.BASELINE_MMA_SYNC, 0, 64, 64, g.F16, A, 64, 1, B, 64, 1, C, 64, g.F16, 1.0, 0.0,
                           None, g.EPI_NONE, stream=0) == 0


def test_q4_validation_without_gpu(g):
    X, W, SB, C = 0x100000, 0x200000, 0x300000, 0x400000
    def call(M=1, N=64, K=128, xd=None, ldx=128, X=X, W=W, SB=SB, cd=None, epi=None, bias=None):
        return g.gemm_q4(M, N, K, g.F16 if xd is None else xd, X, ldx, W, SB, C, N, g.F16 if cd is None else cd,
                         1.0, 0.0, bias, g.EPI_NONE if epi is None else epi, stream=0)
    for kwargs, status in [(dict(K=100), g.ERR_INVALID_ARG),             # K not a multiple of 64
                           (dict(xd=g.F32), g.ERR_UNSUPPORTED),
                           (dict(xd=g.E4M3), g.ERR_UNSUPPORTED),
                           (dict(cd=g.E4M3), g.ERR_UNSUPPORTED),
                           (dict(ldx=100), g.ERR_INVALID_ARG),           # ldx < K
                           (dict(ldx=132), g.ERR_MISALIGNED),            # row pitch not a multiple of 16 bytes
                           (dict(X=X + 2), g.ERR_MISALIGNED),
                           (dict(W=W + 4), g.ERR_MISALIGNED),
                           (dict(epi=g.EPI_BIAS), g.ERR_INVALID_ARG)]:   # bias missing
        with pytest.raises(g.GemmError) as e:
            call(**kwargs)
        assert e.value.status == status, kwargs
    assert call(M=0) == 0 and call(N=0) == 0
    with pytest.raises(g.GemmError) as e:
        g.gemm_q4_dequantize(64, 100, W, SB, C, g.F16, stream=0)
    assert e.value.status == g.ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.gemm_q4_dequantize(64, 128, W, SB, C, g.F32, stream=0)
    assert e.value.status == g.ERR_UNSUPPORTED
    assert g.gemm_q4_dequantize(0, 128, W, SB, C, g.F16, stream=0) == 0


def test_mx_workspace_size_and_validation_without_gpu(g):
    """gemm_mx_workspace_size is a pure function of the sizes; argument errors come back before any
    CUDA call."""
    # MXFP8: 4 blocks of 32 k per 512-byte chunk of 128 rows; MXFP4 rounds chunk columns to pairs
    assert g.gemm_mx_workspace_size(128, 128, 128, g.MX_E4M3) == 512 + 512
    assert g.gemm_mx_workspace_size(4096, 4096, 4096, g.MX_E4M3) == 2 * 32 * 32 * 512
    assert g.gemm_mx_workspace_size(200, 136, 96, g.MX_E4M3) == 2 * 512 + 2 * 512
    assert g.gemm_mx_workspace_size(128, 128, 160, g.MX_E2M1) == 2 * 512 + 2 * 512   # 5 blocks -> 2 chunks
    assert g.gemm_mx_workspace_size(128, 128, 48, g.MX_E4M3) == 0                     # not whole blocks
    assert g.gemm_mx_workspace_size(0, 128, 128, g.MX_E4M3) == 0
    args = (PA, 128, PB, PB, 128, PBIAS, PC, 128)
    for K, cd, elem, status in ((48, g.F32, g.MX_E4M3, g.ERR_INVALID_ARG), (128, g.E4M3, g.MX_E4M3, g.ERR_UNSUPPORTED),
                                (128, g.F32, 7, g.ERR_INVALID_ARG)):
        with pytest.raises(g.GemmError) as ei:
            g.gemm_mx(128, 128, K, elem, *args, cd, 1.0, 0.0, None, g.EPI_NONE, stream=0)
        assert ei.value.status == status
    assert g.gemm_mx(0, 128, 128, g.MX_E4M3, *args, g.F32, 1.0, 0.0, None, g.EPI_NONE, stream=0) == 0   # no-op


def test_q4_ws_workspace_size_and_fallback_without_gpu(g):
    """gemm_q4_workspace_size: 0 below Q4_DEQUANT_ROWS rows of x (the fused kernels run there) or for a
    non-16-bit x, else the 16-bit W rounded to 256 bytes plus gemm()'s own workspace.  gemm_q4_ws without
    a usable workspace is gemm_q4: the same argument errors before any CUDA call."""
    assert g.Q4_DEQUANT_ROWS == 384
    assert g.gemm_q4_workspace_size(383, 4096, 4096, g.F16) == 0
    w = 4096 * 4096 * 2
    assert g.gemm_q4_workspace_size(384, 4096, 4096, g.F16) == w + g.gemm_workspace_size(384, 4096, 4096, g.F16)
    assert g.gemm_q4_workspace_size(4096, 4096, 4096, g.BF16) == w + g.gemm_workspace_size(4096, 4096, 4096, g.BF16)
    assert g.gemm_q4_workspace_size(1000, 100, 192, g.F16) == (100 * 192 * 2 + 255) // 256 * 256 + \
        g.gemm_workspace_size(1000, 100, 192, g.F16)
    assert g.gemm_q4_workspace_size(4096, 4096, 4096, g.F32) == 0
    assert g.gemm_q4_workspace_size(4096, 4096, 100, g.F16) == 0      # K not a multiple of 64
    assert g.gemm_q4_workspace_size(4096, 0, 4096, g.F16) == 0
    X, W, SB, C = 0x100000, 0x200000, 0x300000, 0x400000
    for kw, status in [(dict(K=100), g.ERR_INVALID_ARG), (dict(xd=g.F32), g.ERR_UNSUPPORTED),
                       (dict(ldx=132), g.ERR_MISALIGNED)]:
        K = kw.get("K", 128)
        with pytest.raises(g.GemmError) as e:
            g.gemm_q4_ws(16, 64, K, kw.get("xd", g.F16), X, kw.get("ldx", 128), W, SB, C, 64, g.F16, 1.0, 0.0,
                         None, g.EPI_NONE, workspace=None, workspace_bytes=0, stream=0)
        assert e.value.status == status, kw


def test_binding_fails_loudly_without_the_library(tmp_path):
    """The binding has no fallback: imported where libgemm_gb300.so is absent, it raises ImportError."""
    import shutil
    import subprocess
    import sys
    pkg = tmp_path / "dense_gemm_epilogues_tcgen05_gb300"
    pkg.mkdir()
    shutil.copy(os.path.join(REPO, "dense_gemm_epilogues_tcgen05_gb300", "__init__.py"), pkg / "__init__.py")
    r = subprocess.run([sys.executable, "-c", "import dense_gemm_epilogues_tcgen05_gb300"], cwd=tmp_path,
                       capture_output=True, text=True, env={**os.environ, "PYTHONPATH": str(tmp_path)})
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libgemm_gb300.so is missing" in r.stderr
