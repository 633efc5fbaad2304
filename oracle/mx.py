"""Float64 oracle of the block-scaled (microscaling, "MX") matrix product.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle``: nothing on the product
path imports it, and it shares no code with the CUDA library.

The pages list fp4 and block-scaled MXFP4 next to fp8 among the low-precision
rows of the matrix units (Rigel, section 1) but define neither.  The
definitions used here are those of the OCP Microscaling Formats (MX)
Specification v1.0: a block of 32 consecutive elements shares one scale X, an
E8M0 number (8 exponent bits, bias 127, no sign or fraction; code 0xFF is
NaN), and element i of the block stands for X * P_i, P_i being an FP8 E4M3
(MXFP8) or FP4 E2M1 (MXFP4) number.

Product, with blocks running along K (the contraction), A given as M x K and
B as its transpose, N x K, both K-contiguous (row pitches lda, ldb in
elements):

    a_ik = X^A[i][k // 32] * P^A[i][k]        (exact in float64)
    b_kj = X^B[j][k // 32] * P^B[j][k]
    z_ij = alpha * sum_k a_ik b_kj + beta * c_ij + bias_j
    y_ij = act(z_ij)

with the dense oracle's epilogues, error scale
D_ij = |alpha| sum_k |a_ik||b_kj| + |beta||c_ij| + |bias_j| and per-output-type
tolerances.  Storage: E4M3 elements one per byte; E2M1 elements two per
byte, element k in the low nibble when k is even and in the high nibble when
k is odd (a stated choice: the specification leaves packing to the
implementation); scales one byte each, row-major M x K/32 (A) and N x K/32 (B).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from . import (ACTIVATIONS, EPILOGUES, EPI_NONE, decode, decode_e4m3, fp32_value, max_normalized_error,
               output_values, strided_codes, tolerance)

BLOCK = 32            # elements per shared scale (OCP MX v1.0, section 5)
ELEM_E4M3 = "e4m3"    # MXFP8 (E4M3 elements)
ELEM_E2M1 = "e2m1"    # MXFP4
ELEMENTS = (ELEM_E4M3, ELEM_E2M1)
E2M1_MAX = 6.0
E8M0_NAN = 0xFF


def decode_e2m1(codes) -> np.ndarray:
    """OCP FP4 E2M1: 1 sign, 2 exponent (bias 1), 1 fraction bit; no infinities
    or NaN.  Exponent 0 is subnormal: 0.5 * fraction."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    s, e, m = (c >> 3) & 1, (c >> 1) & 0x3, c & 0x1
    normal = np.ldexp((m + 2).astype(np.float64), (e - 2).astype(np.int32))
    sub = m.astype(np.float64) * 0.5
    val = np.where(e == 0, sub, normal)
    return np.where(s == 1, -val, val)


def decode_e8m0(codes) -> np.ndarray:
    """OCP E8M0 scale: 2^(code - 127) for codes 0..254, NaN for 0xFF."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    val = np.ldexp(np.ones(c.shape, dtype=np.float64), (c - 127).astype(np.int32))
    return np.where(c == E8M0_NAN, np.nan, val)


def element_values(codes: np.ndarray, rows: int, K: int, ld: int, elem: str,
                   row_sel: Optional[np.ndarray] = None) -> np.ndarray:
    """P values (float64) of a rows x K block of K-contiguous elements with row pitch ld
    (in elements), only the rows in row_sel when given."""
    sel = np.arange(rows, dtype=np.int64) if row_sel is None else np.asarray(row_sel, dtype=np.int64)
    flat = np.asarray(codes).reshape(-1)
    if elem == ELEM_E4M3:
        idx = sel[:, None] * ld + np.arange(K, dtype=np.int64)[None, :]
        return decode_e4m3(flat[idx])
    if elem == ELEM_E2M1:
        if ld % 2:
            raise ValueError("E2M1 rows must start on a byte: ld even")
        k = np.arange(K, dtype=np.int64)
        byte = flat[sel[:, None] * (ld // 2) + (k // 2)[None, :]].astype(np.int64)
        nib = np.where((k % 2)[None, :] == 0, byte & 0xF, (byte >> 4) & 0xF)
        return decode_e2m1(nib)
    raise ValueError("unknown element type")


def block_scales(scales: np.ndarray, rows: int, K: int, row_sel: Optional[np.ndarray] = None) -> np.ndarray:
    """X per element (float64), rows x K, from the rows x K/32 scale codes."""
    sel = np.arange(rows, dtype=np.int64) if row_sel is None else np.asarray(row_sel, dtype=np.int64)
    s = np.asarray(scales).reshape(rows, K // BLOCK)[sel]
    return np.repeat(decode_e8m0(s), BLOCK, axis=1)


def mx_reference(M: int, N: int, K: int, elem: str,
                 A: np.ndarray, lda: int, a_scale: np.ndarray,
                 B: np.ndarray, ldb: int, b_scale: np.ndarray,
                 C: Optional[np.ndarray], ldc: int, c_dtype: int,
                 alpha: float, beta: float, bias: Optional[np.ndarray], epilogue: int,
                 rows: Optional[Sequence[int]] = None):
    """Reference output y (float64, not rounded) and error scale D of the MX product.

    A: element codes of the M x K operand (row pitch lda elements); B: those of
    the N x K transposed operand (pitch ldb); a_scale / b_scale: E8M0 codes,
    M x K/32 and N x K/32.  alpha and beta at their binary32 values; beta == 0
    leaves C unread, alpha == 0 or K == 0 leaves A, B and the scales unread.
    Returns (y, D), len(rows) x N (all M rows when rows is None).
    """
    if min(M, N, K) < 0:
        raise ValueError("negative size")
    if K % BLOCK:
        raise ValueError("K must be a multiple of the block size")
    if elem not in ELEMENTS:
        raise ValueError("unknown element type")
    if epilogue not in EPILOGUES:
        raise ValueError("unknown epilogue")
    al, be = fp32_value(alpha), fp32_value(beta)
    row_sel = np.arange(M, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    R = row_sel.size
    z = np.zeros((R, N), dtype=np.float64)
    D = np.zeros((R, N), dtype=np.float64)
    if al != 0.0 and K > 0 and R > 0 and N > 0:
        a = element_values(A, M, K, lda, elem, row_sel) * block_scales(a_scale, M, K, row_sel)   # R x K
        bt = element_values(B, N, K, ldb, elem) * block_scales(b_scale, N, K)                 # N x K
        z += al * (a @ bt.T)
        D += abs(al) * (np.abs(a) @ np.abs(bt).T)
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
    return y, D


def check(problem_args: dict, C_out: np.ndarray, rows: Optional[Sequence[int]] = None) -> dict:
    """An output buffer against the MX reference, at the dense oracle's tolerance
    for the output type (1e-5 for fp32, 2e-3 for 16-bit outputs)."""
    p = problem_args
    y, D = mx_reference(rows=rows, **p)
    out = output_values(C_out, p["M"], p["N"], p["ldc"], p["c_dtype"], rows)
    err = max_normalized_error(out, y, D, p["epilogue"])
    tol = tolerance(-1, p["c_dtype"])
    return {"err": err, "tol": tol, "pass": bool(err <= tol)}
