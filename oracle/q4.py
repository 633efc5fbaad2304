"""Float64 oracle of the 4-bit group-quantized matrix product (decode GEMV).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle``: nothing on the product
path imports it, and it shares no code with the CUDA library.

The pages name quantized matmul -- GEMV for decode, GEMM for prefill, with the
dequantisation fused into the multiply-accumulate -- as the main LLM workload
on Apple GPUs ("X3: Metal GEMM", section 7), but give no storage format.  The
format taken here (a stated choice, the affine group quantization MLX uses):

    W is N x K (output features x input features).  Each group of G = 64
    consecutive k of one row n has a scale s[n][g] and a bias b[n][g], both
    IEEE binary16, and every element a 4-bit code q[n][k] in 0..15:

        W[n][k] = s[n][k // 64] * q[n][k] + b[n][k // 64]

    Storage: q[n][k] is bits 4*(k % 8) .. 4*(k % 8) + 3 of the little-endian
    32-bit word Wq[n * K/8 + k // 8]; scale_bias holds binary16 codes in pairs,
    element 2*(n * K/64 + g) the scale and the next one the bias.

The product follows the dense operation of this library with W^T as B:

    z[m][n] = alpha * sum_k x[m][k] * W[n][k] + beta * c[m][n] + bias[n]
    y[m][n] = act(z[m][n])

and the error scale D[m][n] = |alpha| * sum_k |x[m][k]| |W[n][k]| + |beta||c|
+ |bias| is the dense oracle's, with the same per-output-type tolerances.
Dequantised values are exact in float64 (an 11-bit scale times a 4-bit code
plus an 11-bit bias).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from . import (ACTIVATIONS, EPILOGUES, EPI_NONE, decode, fp32_value, max_normalized_error, output_values,
               strided_codes, tolerance, F16)

GROUP = 64


def unpack_codes(Wq: np.ndarray, N: int, K: int) -> np.ndarray:
    """The N x K 4-bit codes held in the packed words (row n, then k ascending)."""
    if K % 8 != 0:
        raise ValueError("K must be a multiple of 8")
    words = np.asarray(Wq).astype(np.uint64).reshape(N, K // 8)
    shifts = (4 * np.arange(8, dtype=np.uint64))[None, None, :]
    nib = (words[:, :, None] >> shifts) & np.uint64(0xF)
    return nib.reshape(N, K).astype(np.int64)


def dequantize(Wq: np.ndarray, scale_bias: np.ndarray, N: int, K: int) -> np.ndarray:
    """W[n][k] = s[n][k // 64] * q[n][k] + b[n][k // 64] in float64 (N x K)."""
    if K % GROUP != 0:
        raise ValueError("K must be a multiple of the group size 64")
    q = unpack_codes(Wq, N, K).astype(np.float64)
    sb = decode(np.asarray(scale_bias).reshape(-1), F16).reshape(N, K // GROUP, 2)
    s = np.repeat(sb[:, :, 0], GROUP, axis=1)
    b = np.repeat(sb[:, :, 1], GROUP, axis=1)
    return s * q + b


def q4_reference(M: int, N: int, K: int, x_dtype: int, X: np.ndarray, ldx: int,
                 Wq: np.ndarray, scale_bias: np.ndarray,
                 C: Optional[np.ndarray], ldc: int, c_dtype: int,
                 alpha: float, beta: float, bias: Optional[np.ndarray], epilogue: int,
                 rows: Optional[Sequence[int]] = None):
    """Reference output y (float64) and error scale D, len(rows) x N (rows of x / C).

    X holds codes of x_dtype, row m at X[m * ldx ...]; beta == 0 leaves C unread
    and alpha == 0 (or K == 0) leaves x and W unread, as in the dense oracle."""
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
        x = decode(strided_codes(X, M, K, ldx, 1, row_sel), x_dtype)
        W = dequantize(Wq, scale_bias, N, K)
        z += al * (x @ W.T)
        D += abs(al) * (np.abs(x) @ np.abs(W).T)
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
    return (act(z) if act is not None else z), D


def check(problem_args: dict, C_out: np.ndarray, rows: Optional[Sequence[int]] = None) -> dict:
    """Compare an output buffer with the reference: err, tol (by output type) and pass."""
    p = problem_args
    y, D = q4_reference(rows=rows, **p)
    out = output_values(C_out, p["M"], p["N"], p["ldc"], p["c_dtype"], rows)
    err = max_normalized_error(out, y, D, p["epilogue"])
    tol = tolerance(p["x_dtype"], p["c_dtype"])
    return {"err": err, "tol": tol, "pass": bool(err <= tol)}
