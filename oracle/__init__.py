"""Float64 CPU oracle for the dense GEMM with fused epilogue.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may use it.  It shares no code with the CUDA library.

What it computes (the plain definition the kernels reach up to rounding order):

    a_ik = decode(A bytes at i*a_stride_m + k*a_stride_k)        exact in float64
    b_kj = decode(B bytes at k*b_stride_k + j*b_stride_n)
    z_ij = alpha*sum_k a_ik*b_kj + beta*c_ij + bias_j
    y_ij = act(z_ij)                      (bias + activation epilogues)

with act one of GELU (exact erf form), GELU (tanh form), SiLU and ReLU.

Sources on the pages:
  * C = alpha*A*B + beta*C with the epilogue applied to the accumulator before
    the single store -- "Case Study: Steel's BlockMMA" (the paragraph on the
    ending where fusion plugs in: store_result / apply_epilogue) and "Case
    Study: The Tiled GEMM" (the fused alpha*AB + beta*C store).
  * fp32 accumulation regardless of input type -- "Case Study: Steel's
    BlockMMA" (AccumType = float) and Rigel section 2 (accumulator >= fp32).
  * Out-of-range operand elements read as zero, out-of-range outputs never
    written -- "X3: Metal GEMM" sections 2, 4 and 5 (zero fill, masked store).
  * Transposition by strides only -- "Case Study: Steel's BlockMMA" (the
    A_str_m / A_str_k stride constants).
  * The float64 reference over the same quantised bytes, with a per-dtype
    tolerance -- Rigel section 3 ("checksum gate").
  * GELU of bias-added accumulators -- Rigel abstract and section 1
    (GEMM + bias + GELU fusion).  The pages say only "GELU"; the exact erf form
    is the reading taken here.
  * Other activations in the same place -- "Case Study: Steel's BlockMMA"
    (the Epilogue is a pluggable functor applied to every accumulator before
    the store).  Their formulas are the standard definitions: the tanh form of
    GELU (Hendrycks & Gimpel, "Gaussian Error Linear Units", section 2),
    SiLU z*sigmoid(z) (Elfwing, Uchibe & Doya 2018) and ReLU max(z, 0).

The sum over k is taken with a float64 library matmul (a library primitive used
as one step); its rounding error (~K * 2^-53 relative) is nine orders of
magnitude below the tightest tolerance.  Decoders are written from the bit
definitions of IEEE 754 binary16/binary32, bfloat16 (8-bit exponent, 7-bit
fraction) and OCP FP8 E4M3 (bias 7, no infinities, S.1111.111 = NaN).
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np
from scipy.special import erf as _erf
from scipy.special import expit as _expit

# Element type and epilogue codes of the C ABI (restated, not imported).
F32, F16, BF16, E4M3 = 0, 1, 2, 3
EPI_NONE, EPI_BIAS, EPI_BIAS_GELU = 0, 1, 2
EPI_BIAS_GELU_TANH, EPI_BIAS_SILU, EPI_BIAS_RELU = 3, 4, 5
EPILOGUES = (EPI_NONE, EPI_BIAS, EPI_BIAS_GELU, EPI_BIAS_GELU_TANH, EPI_BIAS_SILU, EPI_BIAS_RELU)

# max_z |d/dz GELU(z)|, attained at z = sqrt(2): Phi(sqrt2) + sqrt2*phi(sqrt2).
GELU_LIPSCHITZ = 0.5 * (1.0 + math.erf(1.0)) + math.sqrt(2.0) * math.exp(-1.0) / math.sqrt(2.0 * math.pi)

# Tolerances on the normalised error, keyed by output type (readings recorded
# with the design notes): 16-bit outputs 2e-3, fp32 outputs 1e-5.
TOL_16BIT_OUT = 2e-3
TOL_F32_OUT = 1e-5


# ---------------------------------------------------------------------------
# Bit-level decoders: integer codes -> exact float64 values.
# ---------------------------------------------------------------------------

def _finish(sign, value, nan_mask=None, inf_mask=None):
    out = np.where(sign == 1, -value, value)
    if inf_mask is not None:
        out = np.where(inf_mask, np.where(sign == 1, -np.inf, np.inf), out)
    if nan_mask is not None:
        out = np.where(nan_mask, np.nan, out)
    return out


def decode_f16(codes) -> np.ndarray:
    """IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits."""
    c = np.asarray(codes).astype(np.int64) & 0xFFFF
    s, e, m = (c >> 15) & 1, (c >> 10) & 0x1F, c & 0x3FF
    normal = np.ldexp((m + 1024).astype(np.float64), (e - 25).astype(np.int32))
    sub = np.ldexp(m.astype(np.float64), -24)
    val = np.where(e == 0, sub, normal)
    return _finish(s, val, nan_mask=(e == 0x1F) & (m != 0), inf_mask=(e == 0x1F) & (m == 0))


def decode_bf16(codes) -> np.ndarray:
    """bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits."""
    c = np.asarray(codes).astype(np.int64) & 0xFFFF
    s, e, m = (c >> 15) & 1, (c >> 7) & 0xFF, c & 0x7F
    normal = np.ldexp((m + 128).astype(np.float64), (e - 134).astype(np.int32))
    sub = np.ldexp(m.astype(np.float64), -133)
    val = np.where(e == 0, sub, normal)
    return _finish(s, val, nan_mask=(e == 0xFF) & (m != 0), inf_mask=(e == 0xFF) & (m == 0))


def decode_f32(codes) -> np.ndarray:
    """IEEE binary32: 1 sign, 8 exponent (bias 127), 23 fraction bits."""
    c = np.asarray(codes).astype(np.int64) & 0xFFFFFFFF
    s, e, m = (c >> 31) & 1, (c >> 23) & 0xFF, c & 0x7FFFFF
    normal = np.ldexp((m + (1 << 23)).astype(np.float64), (e - 150).astype(np.int32))
    sub = np.ldexp(m.astype(np.float64), -149)
    val = np.where(e == 0, sub, normal)
    return _finish(s, val, nan_mask=(e == 0xFF) & (m != 0), inf_mask=(e == 0xFF) & (m == 0))


def decode_e4m3(codes) -> np.ndarray:
    """OCP FP8 E4M3: 1 sign, 4 exponent (bias 7), 3 fraction bits; no infinities,
    exponent 1111 with fraction 111 is NaN, every other code is finite."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    s, e, m = (c >> 7) & 1, (c >> 3) & 0xF, c & 0x7
    normal = np.ldexp((m + 8).astype(np.float64), (e - 10).astype(np.int32))
    sub = np.ldexp(m.astype(np.float64), -9)
    val = np.where(e == 0, sub, normal)
    return _finish(s, val, nan_mask=(e == 0xF) & (m == 0x7))


_DECODERS = {F32: decode_f32, F16: decode_f16, BF16: decode_bf16, E4M3: decode_e4m3}


def decode(codes, dtype: int) -> np.ndarray:
    """Decode raw element codes of ``dtype`` to exact float64 values."""
    return _DECODERS[dtype](codes)


def fp32_value(x: float) -> float:
    """The float64 value of the binary32 number the ABI receives for ``x``."""
    with np.errstate(over="ignore"):
        return float(np.float32(x))


# ---------------------------------------------------------------------------
# Operand access through (pointer, stride) views.
# ---------------------------------------------------------------------------

def strided_codes(codes: np.ndarray, rows: int, cols: int, stride_r: int, stride_c: int,
                  row_idx: Optional[Sequence[int]] = None) -> np.ndarray:
    """Codes of the rows x cols matrix whose (r, c) element sits at r*stride_r + c*stride_c.

    Raises if any addressed element lies outside ``codes`` (the oracle never
    reads past a buffer).  ``row_idx`` restricts the result to those rows.
    """
    codes = np.ascontiguousarray(codes).reshape(-1)
    rows_sel = np.arange(rows, dtype=np.int64) if row_idx is None else np.asarray(row_idx, dtype=np.int64)
    if rows_sel.size == 0 or cols == 0:
        return np.zeros((rows_sel.size, cols), dtype=codes.dtype)
    if stride_r < 0 or stride_c < 0:
        raise ValueError("negative strides are not part of the interface")
    last = int(rows_sel.max()) * stride_r + (cols - 1) * stride_c
    if rows_sel.min() < 0 or rows_sel.max() >= rows or last >= codes.size:
        raise IndexError(f"strided view reaches element {last}, buffer has {codes.size}")
    item = codes.itemsize
    full = np.lib.stride_tricks.as_strided(codes, shape=(int(rows_sel.max()) + 1, cols),
                                           strides=(stride_r * item, stride_c * item), writeable=False)
    return np.ascontiguousarray(full[rows_sel])


def gelu(z: np.ndarray) -> np.ndarray:
    """GELU, exact erf form: z * Phi(z) = 0.5*z*(1 + erf(z/sqrt(2)))."""
    return 0.5 * z * (1.0 + _erf(z / math.sqrt(2.0)))


def gelu_tanh(z: np.ndarray) -> np.ndarray:
    """GELU, tanh form: 0.5*z*(1 + tanh(sqrt(2/pi)*(z + 0.044715*z^3)))."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        return 0.5 * z * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (z + 0.044715 * z * z * z)))


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU (swish with beta = 1): z * sigmoid(z) = z / (1 + exp(-z))."""
    z = np.asarray(z, dtype=np.float64)
    return z * _expit(z)


def relu(z: np.ndarray) -> np.ndarray:
    """ReLU: max(z, 0); NaN stays NaN."""
    z = np.asarray(z, dtype=np.float64)
    return np.where(z < 0.0, 0.0, z)


def _max_slope(f, lo: float, hi: float) -> float:
    """max |f'| on [lo, hi] by central differences on a fine grid, refined
    around the best point (the activations here are smooth with one maximum)."""
    z = np.linspace(lo, hi, 200001)
    h = 1e-6
    d = np.abs((f(z + h) - f(z - h)) / (2 * h))
    k = int(np.argmax(d))
    zz = np.linspace(z[max(k - 1, 0)], z[min(k + 1, z.size - 1)], 20001)
    return float(np.max(np.abs((f(zz + h) - f(zz - h)) / (2 * h))))


# max_z |act'(z)| for the activations without a closed form (computed once at
# import; pinned against an independent numerical maximisation in the tests).
GELU_TANH_LIPSCHITZ = _max_slope(gelu_tanh, 0.0, 4.0)
SILU_LIPSCHITZ = _max_slope(silu, 0.0, 6.0)

ACTIVATIONS = {EPI_BIAS_GELU: gelu, EPI_BIAS_GELU_TANH: gelu_tanh, EPI_BIAS_SILU: silu, EPI_BIAS_RELU: relu}


# ---------------------------------------------------------------------------
# The reference result and its per-element error scale.
# ---------------------------------------------------------------------------

def gemm_reference(M: int, N: int, K: int, ab_dtype: int,
                   A: np.ndarray, a_stride_m: int, a_stride_k: int,
                   B: np.ndarray, b_stride_k: int, b_stride_n: int,
                   C: Optional[np.ndarray], ldc: int, c_dtype: int,
                   alpha: float, beta: float,
                   bias: Optional[np.ndarray], epilogue: int,
                   rows: Optional[Sequence[int]] = None,
                   alpha_scale: Optional[np.ndarray] = None, row_scale: Optional[np.ndarray] = None,
                   col_scale: Optional[np.ndarray] = None,
                   residual: Optional[np.ndarray] = None, ldr: int = 0, r_dtype: Optional[int] = None,
                   k_ascending: bool = False):
    """Reference output y (float64, not rounded to the output type) and scale D.

    A, B, C are raw code arrays (flat) in the given element types; ``bias`` is
    a float32 array of length N.  alpha and beta are taken at their binary32
    values, as the ABI passes them.  BLAS conventions: alpha == 0 or K == 0
    leaves A and B unread; beta == 0 leaves C unread.  Returns (y, D), each
    len(rows) x N (all M rows when ``rows`` is None), with

        D_ij = |alpha| * sum_k |a_ik||b_kj| + |beta||c_ij| + |bias_j|.

    Optional product scales (float32 arrays, as the extended call reads them
    from device memory; each absent one is 1): the product term becomes
    alpha * alpha_scale[0] * row_scale[i] * col_scale[j] * sum_k a_ik b_kj,
    and D's first term takes the same factors in absolute value.

    Optional residual (raw codes of an M x ldr row-major array of r_dtype,
    the output type when r_dtype is None): added after the activation,
    y_ij = act(z_ij) + r_ij, the post-activation residual of a transformer
    block; D takes |r_ij| too.

    The sums over k come from a float64 matrix product (BLAS, its own order
    of additions); with ``k_ascending`` they are accumulated one k at a time
    in ascending order instead, the triple loop's order (slow: for small
    cases and for checking that the order moves sums by rounding only).
    """
    if min(M, N, K) < 0:
        raise ValueError("negative size")
    if epilogue not in EPILOGUES:
        raise ValueError("unknown epilogue")
    al, be = fp32_value(alpha), fp32_value(beta)
    row_sel = np.arange(M, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    R = row_sel.size
    z = np.zeros((R, N), dtype=np.float64)
    D = np.zeros((R, N), dtype=np.float64)
    if al != 0.0 and K > 0 and R > 0 and N > 0:
        a = decode(strided_codes(A, M, K, a_stride_m, a_stride_k, row_sel), ab_dtype)
        b = decode(strided_codes(B, K, N, b_stride_k, b_stride_n), ab_dtype)
        f = al if alpha_scale is None else al * float(np.asarray(alpha_scale, np.float32).reshape(-1)[0])
        fac = np.full((R, N), f, dtype=np.float64)
        if row_scale is not None:
            fac *= np.asarray(row_scale, np.float32).astype(np.float64).reshape(-1)[row_sel][:, None]
        if col_scale is not None:
            fac *= np.asarray(col_scale, np.float32).astype(np.float64).reshape(-1)[None, :N]
        if k_ascending:
            ab, aabs = np.zeros((R, N)), np.zeros((R, N))
            for k in range(K):
                ab += a[:, k, None] * b[None, k, :]
                aabs += np.abs(a[:, k, None]) * np.abs(b[None, k, :])
        else:
            ab, aabs = a @ b, np.abs(a) @ np.abs(b)
        z += fac * ab
        D += np.abs(fac) * aabs
    if be != 0.0 and R > 0 and N > 0:
        c = decode(strided_codes(C, M, N, ldc, 1, row_sel), c_dtype)
        z += be * c
        D += abs(be) * np.abs(c)
    if epilogue != EPI_NONE:
        bvals = np.asarray(bias, dtype=np.float32).astype(np.float64).reshape(-1)
        if bvals.size != N:
            raise ValueError("bias must hold N values")
        z += bvals[None, :]
        D += np.abs(bvals)[None, :]
    act = ACTIVATIONS.get(epilogue)
    y = act(z) if act is not None else z
    if residual is not None and R > 0 and N > 0:
        r = decode(strided_codes(residual, M, N, ldr, 1, row_sel), c_dtype if r_dtype is None else r_dtype)
        y = y + r
        D += np.abs(r)
    return y, D


def lipschitz(epilogue: int) -> float:
    """max |act'| of the epilogue's activation (1 without one): how far an
    error in z can move the output."""
    return {EPI_BIAS_GELU: GELU_LIPSCHITZ, EPI_BIAS_GELU_TANH: GELU_TANH_LIPSCHITZ,
            EPI_BIAS_SILU: SILU_LIPSCHITZ}.get(epilogue, 1.0)


def normalized_error(out: np.ndarray, ref: np.ndarray, D: np.ndarray, epilogue: int) -> np.ndarray:
    """Per-element |out - ref| / scale, scale = D times max|act'| (1 without an activation).

    Where the scale is 0 the reference is exact and any difference is
    infinite error; NaN anywhere in ``out`` counts as infinite error.
    """
    scale = D * lipschitz(epilogue)
    diff = np.abs(np.asarray(out, dtype=np.float64) - ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(scale > 0, diff / np.where(scale > 0, scale, 1.0), np.where(diff == 0, 0.0, np.inf))
    return np.where(np.isnan(r), np.inf, r)


def max_normalized_error(out, ref, D, epilogue) -> float:
    r = normalized_error(out, ref, D, epilogue)
    return float(r.max()) if r.size else 0.0


def tolerance(ab_dtype: int, c_dtype: int) -> float:
    """2e-3 for 16-bit outputs; 1e-5 for fp32 outputs (fp32 and fp8 inputs included)."""
    return TOL_16BIT_OUT if c_dtype in (F16, BF16) else TOL_F32_OUT


def output_values(C_out: np.ndarray, M: int, N: int, ldc: int, c_dtype: int,
                  rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """Decode the M x N result held in an M x ldc row-major output buffer."""
    return decode(strided_codes(C_out, M, N, ldc, 1, rows), c_dtype)


def check(problem_args: dict, C_out: np.ndarray, rows: Optional[Sequence[int]] = None) -> dict:
    """Compare an output buffer with the reference; returns err, tol and pass."""
    p = problem_args
    y, D = gemm_reference(rows=rows, **p)
    out = output_values(C_out, p["M"], p["N"], p["ldc"], p["c_dtype"], rows)
    err = max_normalized_error(out, y, D, p["epilogue"])
    tol = tolerance(p["ab_dtype"], p["c_dtype"])
    return {"err": err, "tol": tol, "pass": bool(err <= tol)}


# ---------------------------------------------------------------------------
# fp8 E4M3 outputs and the amax reduction (gemm_ex).
# ---------------------------------------------------------------------------
E4M3_MAX = 448.0
FP8_OUT_REL = 2.0 ** -4   # half a unit in the last place of a 3-bit fraction, relative to |value|
FP8_OUT_ABS = 2.0 ** -10  # half the subnormal step 2^-9


def fp8_output_error(out_values: np.ndarray, ref: np.ndarray, D: np.ndarray, out_scale: float,
                     epilogue: int) -> np.ndarray:
    """Per-element error of an E4M3 output that encodes y / out_scale (saturating at 448).

    The output must be y/s rounded to a representable E4M3 value: saturate the
    reference to +-448 s, allow the rounding of a 3-bit fraction (2^-4 of the
    value, or 2^-10 s among subnormals), and measure what is left over in units
    of the accumulation's error scale D (times max|act'|), as for other outputs."""
    s = fp32_value(out_scale)
    yc = np.clip(ref, -E4M3_MAX * s, E4M3_MAX * s)
    got = np.asarray(out_values, dtype=np.float64) * s
    excess = np.maximum(np.abs(got - yc) - (FP8_OUT_REL * np.abs(yc) + FP8_OUT_ABS * s), 0.0)
    scale = D * lipschitz(epilogue)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(scale > 0, excess / np.where(scale > 0, scale, 1.0), np.where(excess == 0, 0.0, np.inf))
    return np.where(np.isnan(got), np.inf, r)


def check_fp8_output(problem_args: dict, C_out: np.ndarray, out_scale: float,
                     rows: Optional[Sequence[int]] = None) -> dict:
    """An E4M3 output buffer against the reference: the rounding allowance of
    fp8_output_error, then the 16-bit-output tolerance on what remains."""
    p = problem_args
    y, D = gemm_reference(rows=rows, **p)
    out = output_values(C_out, p["M"], p["N"], p["ldc"], E4M3, rows)
    r = fp8_output_error(out, y, D, out_scale, p["epilogue"])
    err = float(r.max()) if r.size else 0.0
    return {"err": err, "tol": TOL_16BIT_OUT, "pass": bool(err <= TOL_16BIT_OUT)}


def amax_reference(problem_args: dict):
    """max over all outputs of |y| (the activated value before any output scaling
    or cast) and the error scale D's largest value, which bounds how far an
    fp32-accumulated maximum may differ (its allowance is TOL_F32_OUT * that)."""
    y, D = gemm_reference(**problem_args)
    if y.size == 0:
        return 0.0, 0.0
    return float(np.abs(y).max()), float((D * lipschitz(problem_args["epilogue"])).max())
