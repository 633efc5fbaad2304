"""Python binding of the GB300 dense GEMM + fused-epilogue library.

Argument marshalling only: every call goes straight to the C ABI in
``libgemm_gb300.so`` (declared in ``include/gemm_gb300.h``); all arithmetic
runs in that library's CUDA kernels.  Buffers may be given as torch tensors
(their ``data_ptr()`` is passed) or as raw integer addresses.  PyTorch is used
only for device memory and streams.

Importing this package fails loudly (ImportError) when the library has not
been built; build it with ``python dense_gemm_epilogues_tcgen05_gb300/build.py``.
"""
from __future__ import annotations

import ctypes
import os

import torch  # noqa: F401  (loads the CUDA runtime the library links against)

__all__ = [
    "F32", "F16", "BF16", "E4M3",
    "EPI_NONE", "EPI_BIAS", "EPI_BIAS_GELU", "EPI_BIAS_GELU_TANH", "EPI_BIAS_SILU", "EPI_BIAS_RELU",
    "PATH_NOOP", "PATH_EPILOGUE_ONLY", "PATH_TCGEN05", "PATH_SIMT",
    "TILE_AUTO", "TILE_1SM_256", "TILE_1SM_128", "TILE_PAIR",
    "GemmError", "gemm", "gemm_query_path", "gemm_workspace_size", "gemm_bias_gelu",
    "SCHED_AUTO", "SCHED_TILES", "SCHED_STREAM_K", "ORDER_AUTO", "ORDER_AS_GIVEN", "ORDER_TRANSPOSED",
    "gemm_set_operand_order", "MCAST_AUTO", "MCAST_OFF", "MCAST_ON", "gemm_set_multicast", "gemm_last_launch",
    "BASELINE_SIMT", "BASELINE_MMA_SYNC", "gemm_baseline", "gemm_q4", "gemm_q4_dequantize", "Q4_MAX_ROWS",
    "gemm_q4_ws", "gemm_q4_workspace_size", "Q4_DEQUANT_ROWS",
    "Q4_AUTO", "Q4_FFMA", "Q4_MMA", "gemm_set_q4_kernel",
    "gemm_ex", "gemm_get_tuning", "MX_E4M3", "MX_E2M1", "gemm_mx", "gemm_mx_workspace_size",
    "gemm_set_tile_policy", "gemm_query_tile", "gemm_set_schedule", "gemm_builtin_scratch", "gemm_wait_selftest",
    "gemm_device_status", "gemm_status_string", "gemm_version", "LIB_PATH", "lib",
]

# gemm_dtype_t
F32, F16, BF16, E4M3 = 0, 1, 2, 3
# gemm_epilogue_t
EPI_NONE, EPI_BIAS, EPI_BIAS_GELU, EPI_BIAS_GELU_TANH, EPI_BIAS_SILU, EPI_BIAS_RELU = 0, 1, 2, 3, 4, 5
# gemm_path_t
PATH_NOOP, PATH_EPILOGUE_ONLY, PATH_TCGEN05, PATH_SIMT = 0, 1, 2, 3
# gemm_tile_policy_t
TILE_AUTO, TILE_1SM_256, TILE_1SM_128, TILE_PAIR = 0, 1, 2, 3
# gemm_schedule_t
SCHED_AUTO, SCHED_TILES, SCHED_STREAM_K = 0, 1, 2
# gemm_operand_order_t
ORDER_AUTO, ORDER_AS_GIVEN, ORDER_TRANSPOSED = 0, 1, 2
# gemm_multicast_t
MCAST_AUTO, MCAST_OFF, MCAST_ON = 0, 1, 2
# gemm_baseline_t
BASELINE_SIMT, BASELINE_MMA_SYNC = 0, 1
# rows of x the decode kernels take; gemm_q4 runs the fused prefill beyond
Q4_MAX_ROWS = 8
Q4_DEQUANT_ROWS = 384  # GEMM_Q4_DEQUANT_ROWS: from this many rows of x gemm_q4_ws expands W once
# gemm_q4_kernel_t
Q4_AUTO, Q4_FFMA, Q4_MMA = 0, 1, 2
# gemm_mx_elem_t
MX_E4M3, MX_E2M1 = 0, 1
# gemm_status_t
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(7)

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgemm_gb300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python dense_gemm_epilogues_tcgen05_gb300/build.py` (nvcc, sm_103a)")

lib = ctypes.CDLL(LIB_PATH)

_i64, _f32, _vp, _int, _sz = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t

lib.gemm.restype = _int
lib.gemm.argtypes = [_i64, _i64, _i64, _int, _vp, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _int,
                     _f32, _f32, _vp, _int, _vp, _sz, _vp]
lib.gemm_query_path.restype = _int
lib.gemm_query_path.argtypes = [_i64, _i64, _i64, _int, _vp, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _int,
                                _f32, _f32, _vp, _int, ctypes.POINTER(_int)]
lib.gemm_workspace_size.restype = _sz
lib.gemm_workspace_size.argtypes = [_i64, _i64, _i64, _int]
lib.gemm_bias_gelu.restype = _int
lib.gemm_bias_gelu.argtypes = [_i64, _i64, _vp, _i64, _int, _vp, _vp]
lib.gemm_set_tile_policy.restype = _int
lib.gemm_set_tile_policy.argtypes = [_int, _int]
lib.gemm_query_tile.restype = _int
lib.gemm_query_tile.argtypes = [_i64, _i64, _i64, _int, _int, ctypes.POINTER(_int), ctypes.POINTER(_int),
                                ctypes.POINTER(_int)]
lib.gemm_builtin_scratch.restype = _int
lib.gemm_builtin_scratch.argtypes = [_i64, _i64, _i64, _int, _vp, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _int,
                                     _f32, _f32, _vp, _int, _vp]
lib.gemm_wait_selftest.restype = _int
lib.gemm_wait_selftest.argtypes = [_vp, ctypes.c_uint64, _vp]
lib.gemm_set_schedule.restype = _int
lib.gemm_set_schedule.argtypes = [_int]
lib.gemm_set_operand_order.restype = _int
lib.gemm_set_operand_order.argtypes = [_int]
lib.gemm_set_multicast.restype = _int
lib.gemm_set_multicast.argtypes = [_int]


class _LaunchInfo(ctypes.Structure):
    """gemm_launch_info_t"""
    _fields_ = [(n, _int) for n in ("path", "kind", "bn", "transposed", "cluster_ctas", "grid_ctas", "tiles",
                                    "stream_k_tiles", "tf32x3")]


lib.gemm_last_launch.restype = _int
lib.gemm_last_launch.argtypes = [ctypes.POINTER(_LaunchInfo)]
class _Scales(ctypes.Structure):
    """gemm_scales_t"""
    _fields_ = [("alpha_scale", ctypes.c_void_p), ("row_scale", ctypes.c_void_p), ("col_scale", ctypes.c_void_p),
                ("out_scale", ctypes.c_void_p), ("amax", ctypes.c_void_p), ("residual", ctypes.c_void_p),
                ("ldr", ctypes.c_int64)]


lib.gemm_ex.restype = _int
lib.gemm_ex.argtypes = [_i64, _i64, _i64, _int, _vp, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _int,
                        _f32, _f32, _vp, _int, ctypes.POINTER(_Scales), _vp, _sz, _vp]
lib.gemm_set_q4_kernel.restype = _int
lib.gemm_set_q4_kernel.argtypes = [_int]


class _Tuning(ctypes.Structure):
    """gemm_tuning_t"""
    _fields_ = [(n, _int) for n in ("tile_policy", "tile_bn", "schedule", "operand_order", "multicast",
                                    "q4_kernel")]


lib.gemm_get_tuning.restype = _int
lib.gemm_get_tuning.argtypes = [ctypes.POINTER(_Tuning)]
lib.gemm_q4.restype = _int
lib.gemm_q4.argtypes = [_i64, _i64, _i64, _int, ctypes.c_void_p, _i64, ctypes.c_void_p, ctypes.c_void_p,
                        ctypes.c_void_p, _i64, _int, ctypes.c_float, ctypes.c_float, ctypes.c_void_p, _int,
                        ctypes.c_void_p]
lib.gemm_q4_ws.restype = _int
lib.gemm_q4_ws.argtypes = [_i64, _i64, _i64, _int, ctypes.c_void_p, _i64, ctypes.c_void_p, ctypes.c_void_p,
                           ctypes.c_void_p, _i64, _int, ctypes.c_float, ctypes.c_float, ctypes.c_void_p, _int,
                           ctypes.c_void_p, _sz, ctypes.c_void_p]
lib.gemm_q4_workspace_size.restype = _sz
lib.gemm_q4_workspace_size.argtypes = [_i64, _i64, _i64, _int]
lib.gemm_q4_dequantize.restype = _int
lib.gemm_q4_dequantize.argtypes = [_i64, _i64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, _int,
                                   ctypes.c_void_p]
lib.gemm_baseline.restype = _int
lib.gemm_baseline.argtypes = [_int, _i64, _i64, _i64, _int, ctypes.c_void_p, _i64, _i64, ctypes.c_void_p, _i64, _i64,
                              ctypes.c_void_p, _i64, _int, ctypes.c_float, ctypes.c_float, ctypes.c_void_p, _int,
                              ctypes.c_void_p]
lib.gemm_mx.restype = _int
lib.gemm_mx.argtypes = [_i64, _i64, _i64, _int, _vp, _i64, _vp, _vp, _i64, _vp, _vp, _i64, _int, _f32, _f32, _vp,
                        _int, _vp, _sz, _vp]
lib.gemm_mx_workspace_size.restype = _sz
lib.gemm_mx_workspace_size.argtypes = [_i64, _i64, _i64, _int]
lib.gemm_device_status.restype = _int
lib.gemm_device_status.argtypes = [_vp]
lib.gemm_status_string.restype = ctypes.c_char_p
lib.gemm_status_string.argtypes = [_int]
lib.gemm_version.restype = ctypes.c_char_p
lib.gemm_version.argtypes = []


class GemmError(RuntimeError):
    """A non-OK gemm_status_t; ``.status`` holds the code."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gemm_status_string(status)} (status {status})")


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    raise TypeError(f"expected a torch.Tensor, an int address or None, got {type(x).__name__}")


def _stream(s):
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str) -> int:
    if status != OK:
        raise GemmError(status, where)
    return status


def gemm(M, N, K, ab_dtype, A, a_stride_m, a_stride_k, B, b_stride_k, b_stride_n, C, ldc, c_dtype,
         alpha, beta, bias, epilogue, workspace=None, workspace_bytes=0, stream=None) -> int:
    """C = cast(epilogue(alpha*A*B + beta*C + bias)) on the GPU; see include/gemm_gb300.h.

    ``stream`` defaults to PyTorch's current stream.  Raises GemmError on a
    non-OK status; returns 0 once the work is enqueued.
    """
    st = lib.gemm(M, N, K, ab_dtype, _ptr(A), a_stride_m, a_stride_k, _ptr(B), b_stride_k, b_stride_n,
                  _ptr(C), ldc, c_dtype, alpha, beta, _ptr(bias), epilogue, _ptr(workspace), workspace_bytes,
                  _stream(stream))
    return _check(st, "gemm")


def gemm_builtin_scratch(M, N, K, ab_dtype, A, a_stride_m, a_stride_k, B, b_stride_k, b_stride_n, C, ldc,
                         c_dtype, alpha, beta, bias, epilogue, stream=None) -> int:
    """gemm() without a workspace argument, for callers that cannot allocate device
    memory: the stream-K scratch comes from the library's fixed device array (see
    include/gemm_gb300.h for its size and the rules on overlapping calls)."""
    st = lib.gemm_builtin_scratch(M, N, K, ab_dtype, _ptr(A), a_stride_m, a_stride_k, _ptr(B), b_stride_k,
                                  b_stride_n, _ptr(C), ldc, c_dtype, alpha, beta, _ptr(bias), epilogue,
                                  _stream(stream))
    return _check(st, "gemm_builtin_scratch")


def gemm_query_path(M, N, K, ab_dtype, A, a_stride_m, a_stride_k, B, b_stride_k, b_stride_n, C, ldc, c_dtype,
                    alpha, beta, bias, epilogue) -> int:
    """Which kernel family gemm() would run for these arguments (PATH_*); launches nothing."""
    out = _int(-1)
    st = lib.gemm_query_path(M, N, K, ab_dtype, _ptr(A), a_stride_m, a_stride_k, _ptr(B), b_stride_k,
                             b_stride_n, _ptr(C), ldc, c_dtype, alpha, beta, _ptr(bias), epilogue,
                             ctypes.byref(out))
    _check(st, "gemm_query_path")
    return out.value


def gemm_workspace_size(M, N, K, ab_dtype) -> int:
    return int(lib.gemm_workspace_size(M, N, K, ab_dtype))


def gemm_bias_gelu(M, N, C, ldc, c_dtype, bias, stream=None) -> int:
    """Unfused pass C = cast(GELU(C + bias)) (measurement of what fusion saves)."""
    return _check(lib.gemm_bias_gelu(M, N, _ptr(C), ldc, c_dtype, _ptr(bias), _stream(stream)),
                  "gemm_bias_gelu")


def gemm_set_tile_policy(policy, bn=0) -> int:
    """The calling thread's tile policy of the tcgen05 path (TILE_*); bn only with TILE_PAIR."""
    return _check(lib.gemm_set_tile_policy(policy, bn), "gemm_set_tile_policy")


def gemm_set_schedule(schedule) -> int:
    """The calling thread's schedule of the pair kernel (SCHED_*)."""
    return _check(lib.gemm_set_schedule(schedule), "gemm_set_schedule")


def gemm_set_operand_order(order) -> int:
    """The calling thread's operand order of the pair kernel (ORDER_*): whether it may compute C^T = B^T A^T."""
    return _check(lib.gemm_set_operand_order(order), "gemm_set_operand_order")


def gemm_set_multicast(mode) -> int:
    """The calling thread's cluster shape of the pair kernel (MCAST_*): two SM pairs sharing A by TMA
    multicast (only over this device's own memory), or one."""
    return _check(lib.gemm_set_multicast(mode), "gemm_set_multicast")


def gemm_baseline(kind, M, N, K, ab_dtype, A, a_stride_m, a_stride_k, B, b_stride_k, b_stride_n, C, ldc, c_dtype,
                  alpha, beta, bias, epilogue, stream=None) -> int:
    """The same operation as gemm() on a baseline kernel of the cheap-baseline gate (BASELINE_*)."""
    st = lib.gemm_baseline(kind, M, N, K, ab_dtype, _ptr(A), a_stride_m, a_stride_k, _ptr(B), b_stride_k, b_stride_n,
                           _ptr(C), ldc, c_dtype, alpha, beta, _ptr(bias), epilogue, _stream(stream))
    return _check(st, "gemm_baseline")


def gemm_ex(M, N, K, ab_dtype, A, a_stride_m, a_stride_k, B, b_stride_k, b_stride_n, C, ldc, c_dtype,
            alpha, beta, bias, epilogue, alpha_scale=None, row_scale=None, col_scale=None, out_scale=None,
            amax=None, residual=None, ldr=0, workspace=None, workspace_bytes=0, stream=None) -> int:
    """gemm() with scales (device fp32 arrays: alpha_scale[1], row_scale[M], col_scale[N], out_scale[1] for
    an E4M3 output, amax[1] raised to max |y|) and a post-activation residual (M x ldr array of the output
    type, added after the activation); None = absent."""
    sc = _Scales(_ptr(alpha_scale), _ptr(row_scale), _ptr(col_scale), _ptr(out_scale), _ptr(amax),
                 _ptr(residual), ldr)
    st = lib.gemm_ex(M, N, K, ab_dtype, _ptr(A), a_stride_m, a_stride_k, _ptr(B), b_stride_k, b_stride_n,
                     _ptr(C), ldc, c_dtype, alpha, beta, _ptr(bias), epilogue, ctypes.byref(sc), _ptr(workspace),
                     workspace_bytes, _stream(stream))
    return _check(st, "gemm_ex")


def gemm_set_q4_kernel(kind) -> int:
    """The calling thread's kernel of gemm_q4 (Q4_*): AUTO, the CUDA-core kernel, or the tensor-core one."""
    return _check(lib.gemm_set_q4_kernel(kind), "gemm_set_q4_kernel")


def gemm_q4(M, N, K, x_dtype, X, ldx, Wq, scale_bias, C, ldc, c_dtype, alpha, beta, bias, epilogue,
            stream=None) -> int:
    """C = cast(epilogue(alpha * x W^T + beta*C + bias)) with 4-bit group-quantized W: decode kernels for
    M <= 8 rows of x, the tensor-core prefill kernel (dequantisation fused in) beyond."""
    st = lib.gemm_q4(M, N, K, x_dtype, _ptr(X), ldx, _ptr(Wq), _ptr(scale_bias), _ptr(C), ldc, c_dtype, alpha,
                     beta, _ptr(bias), epilogue, _stream(stream))
    return _check(st, "gemm_q4")


def gemm_q4_ws(M, N, K, x_dtype, X, ldx, Wq, scale_bias, C, ldc, c_dtype, alpha, beta, bias, epilogue,
               workspace=None, workspace_bytes=0, stream=None) -> int:
    """gemm_q4 with a workspace: from Q4_DEQUANT_ROWS rows of x, W is expanded once into the workspace and
    multiplied by the dense kernel (faster for long prompts); otherwise gemm_q4."""
    st = lib.gemm_q4_ws(M, N, K, x_dtype, _ptr(X), ldx, _ptr(Wq), _ptr(scale_bias), _ptr(C), ldc, c_dtype, alpha,
                        beta, _ptr(bias), epilogue, _ptr(workspace), workspace_bytes, _stream(stream))
    return _check(st, "gemm_q4_ws")


def gemm_q4_workspace_size(M, N, K, x_dtype) -> int:
    """Bytes of workspace gemm_q4_ws uses for this shape (0: it runs the fused kernels)."""
    return int(lib.gemm_q4_workspace_size(M, N, K, x_dtype))


def gemm_q4_dequantize(N, K, Wq, scale_bias, W, w_dtype, stream=None) -> int:
    """W = round(s*q + b) as an N x K row-major fp16 / bf16 array (prefill: then gemm())."""
    st = lib.gemm_q4_dequantize(N, K, _ptr(Wq), _ptr(scale_bias), _ptr(W), w_dtype, _stream(stream))
    return _check(st, "gemm_q4_dequantize")


def gemm_get_tuning() -> dict:
    """The calling thread's tuning settings (gemm_tuning_t as a dict)."""
    t = _Tuning()
    _check(lib.gemm_get_tuning(ctypes.byref(t)), "gemm_get_tuning")
    return {n: getattr(t, n) for n, _ in _Tuning._fields_}


def gemm_mx(M, N, K, elem, A, lda, a_scale, B, ldb, b_scale, C, ldc, c_dtype, alpha, beta, bias, epilogue,
            workspace=None, workspace_bytes=0, stream=None) -> int:
    """Block-scaled product (MX_E4M3 / MX_E2M1 elements, E8M0 scales per 32 k): A M x K, B given as its
    transpose N x K, both K-contiguous; see include/gemm_gb300.h."""
    st = lib.gemm_mx(M, N, K, elem, _ptr(A), lda, _ptr(a_scale), _ptr(B), ldb, _ptr(b_scale), _ptr(C), ldc, c_dtype,
                     alpha, beta, _ptr(bias), epilogue, _ptr(workspace), workspace_bytes, _stream(stream))
    return _check(st, "gemm_mx")


def gemm_mx_workspace_size(M, N, K, elem) -> int:
    return int(lib.gemm_mx_workspace_size(M, N, K, elem))


def gemm_last_launch() -> dict:
    """What this thread's last successful gemm() enqueued (gemm_launch_info_t as a dict)."""
    info = _LaunchInfo()
    _check(lib.gemm_last_launch(ctypes.byref(info)), "gemm_last_launch")
    return {n: getattr(info, n) for n, _ in _LaunchInfo._fields_}


def gemm_query_tile(M, N, K, ab_dtype, c_dtype):
    """(kind, bn, units) of the tcgen05 path on the current device: kind 1 = one SM per
    tile, 2 = SM pair; units = tiles in flight at once (CTAs or clusters)."""
    kind, bn, units = _int(0), _int(0), _int(0)
    _check(lib.gemm_query_tile(M, N, K, ab_dtype, c_dtype, ctypes.byref(kind), ctypes.byref(bn),
                               ctypes.byref(units)), "gemm_query_tile")
    return kind.value, bn.value, units.value


def gemm_device_status(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device status as a gemm_status_t code."""
    return int(lib.gemm_device_status(_stream(stream)))


def gemm_wait_selftest(never_set, limit_ns, stream=None) -> int:
    """Run the bounded-wait self-test (see include/gemm_gb300.h); then gemm_device_status()."""
    return _check(lib.gemm_wait_selftest(_ptr(never_set), limit_ns, _stream(stream)), "gemm_wait_selftest")


def gemm_status_string(status: int) -> str:
    return lib.gemm_status_string(status).decode()


def gemm_version() -> str:
    return lib.gemm_version().decode()
