"""Pins of the quantized-matmul oracle (oracle.q4) against things other than itself:

* the storage format written out by hand (nibble order, scale/bias pairs);
* packing by the independent packer in ``workloads`` round-tripping;
* exact rational brute force from the raw words, in plain Python integers;
* a closed form (all codes zero: W is the group bias);
* agreement with the dense oracle on the dequantised matrix, which is pinned
  on its own;
* planted mistakes (nibble order, group size, dropped bias, transposed W)
  all flagged by the error metric.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from oracle import q4


def test_unpack_follows_the_stated_format():
    words = np.array([0x76543210, 0xFEDCBA98], dtype=np.uint32)
    assert q4.unpack_codes(words, 1, 16).tolist() == [list(range(16))]
    # one nibble set at a time: code j lands at k = j
    for j in range(8):
        w = np.array([0xF << (4 * j)], dtype=np.uint32)
        codes = q4.unpack_codes(w, 1, 8)[0]
        assert codes.tolist() == [15 if k == j else 0 for k in range(8)]


def test_pack_and_unpack_round_trip():
    g = torch.Generator().manual_seed(3)
    q = torch.randint(0, 16, (5, 192), generator=g)
    words = wl.pack_q4(q)
    assert words.dtype == torch.int32 and words.numel() == 5 * 192 // 8
    assert np.array_equal(q4.unpack_codes(words.numpy(), 5, 192), q.numpy())


def test_dequantize_by_hand():
    # scale 0.5 (binary16 0x3800) and bias -2 (0xC000) for the only group; codes 0..15 then 3s
    codes = list(range(16)) + [3] * 48
    words = np.array([sum(codes[8 * w + j] << (4 * j) for j in range(8)) for w in range(8)], dtype=np.uint32)
    sb = np.array([0x3800, 0xC000], dtype=np.uint16)
    W = q4.dequantize(words, sb, 1, 64)
    assert W[0, :16].tolist() == [0.5 * c - 2.0 for c in range(16)]
    assert W[0, 16:].tolist() == [-0.5] * 48


def _half(code):
    """binary16 code -> Fraction, from the bit definition (normal and subnormal)."""
    s = -1 if code & 0x8000 else 1
    e, f = (code >> 10) & 0x1F, code & 0x3FF
    assert e != 31
    if e == 0:
        return s * Fraction(f, 1 << 24)
    return s * Fraction(1024 + f, 1 << 10) * Fraction(2) ** (e - 15)


@pytest.mark.parametrize("M,N,K", [(1, 1, 64), (2, 3, 128), (3, 5, 192)])
def test_brute_force_exact(M, N, K):
    p = wl.q4_problem(11 + M + N + K, M, N, K, wl.F16, wl.F32, alpha=1.0, beta=0.0, integer=True)
    words = [int(v) & 0xFFFFFFFF for v in p.Wq.numpy().tolist()]
    sb = [int(v) & 0xFFFF for v in p.SB.numpy().tolist()]
    xs = [_half(int(v) & 0xFFFF) for v in p.X.view(torch.int16).numpy().tolist()]
    y, _ = q4.q4_reference(**p.oracle_args())
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                code = (words[n * K // 8 + k // 8] >> (4 * (k % 8))) & 0xF
                g = n * K // 64 + k // 64
                w = _half(sb[2 * g]) * code + _half(sb[2 * g + 1])
                acc += xs[m * K + k] * w
            assert Fraction(y[m, n]) == acc


def test_zero_codes_leave_the_group_bias():
    p = wl.q4_problem(5, 2, 4, 128, wl.F16, wl.F32, alpha=0.5, integer=True)
    p.Wq.zero_()
    y, D = q4.q4_reference(**p.oracle_args())
    x = oracle.decode(p.X.view(torch.int16).numpy(), wl.F16).reshape(2, 128)
    sb = oracle.decode(p.SB.numpy(), wl.F16).reshape(4, 2, 2)
    want = 0.5 * np.stack([x[:, :64].sum(1)[:, None] * sb[None, :, 0, 1] +
                           x[:, 64:].sum(1)[:, None] * sb[None, :, 1, 1]])[0]
    assert np.array_equal(y, want)


@pytest.mark.parametrize("epi", [wl.EPI_NONE, wl.EPI_BIAS_GELU])
def test_matches_the_dense_oracle_on_the_dequantised_matrix(epi):
    p = wl.q4_problem(21, 3, 24, 256, wl.BF16, wl.F32, alpha=0.75, beta=0.5, epilogue=epi, integer=True)
    a = p.oracle_args()
    y, D = q4.q4_reference(**a)
    W = q4.dequantize(a["Wq"], a["scale_bias"], 24, 256)            # integers: exact in fp32
    x = oracle.decode(a["X"], wl.BF16)                               # bf16 values: exact in fp32
    Bf = W.astype(np.float32).view(np.int32).reshape(-1)             # W^T as B with b_stride_k = 1, b_stride_n = K
    Af = x.astype(np.float32).view(np.int32)
    y2, D2 = oracle.gemm_reference(3, 24, 256, wl.F32, Af, 256, 1, Bf, 1, 256, a["C"], a["ldc"], a["c_dtype"],
                                   a["alpha"], a["beta"], a["bias"], epi)
    assert np.array_equal(y, y2) and np.array_equal(D, D2)


@pytest.mark.parametrize("mistake", ["nibble_order", "group_32", "no_bias", "transposed"])
def test_planted_mistakes_are_flagged(mistake):
    p = wl.q4_problem(31, 4, 32, 256, wl.F16, wl.F32)
    a = p.oracle_args()
    y, D = q4.q4_reference(**a)
    N, K = 32, 256
    codes = q4.unpack_codes(a["Wq"], N, K)
    sb = oracle.decode(a["scale_bias"], wl.F16).reshape(N, K // 64, 2)
    if mistake == "nibble_order":
        codes = codes.reshape(N, K // 8, 8)[:, :, ::-1].reshape(N, K)
    if mistake == "group_32":
        # scales and biases read as if a group held 32 values (the last group stretched)
        gi = np.minimum(np.arange(K) // 32, K // 64 - 1)
        W = sb[:, gi, 0] * codes + sb[:, gi, 1]
    else:
        s = np.repeat(sb[:, :, 0], 64, axis=1)
        b = np.repeat(sb[:, :, 1], 64, axis=1)
        W = s * codes + (0 if mistake == "no_bias" else b)
    x = oracle.decode(a["X"], wl.F16).reshape(4, K)
    out = x @ (W.T if mistake != "transposed" else W.reshape(K, N))
    err = oracle.max_normalized_error(out.astype(np.float32), y, D, wl.EPI_NONE)
    assert err > oracle.tolerance(wl.F16, wl.F32)
    # and the faithful computation passes, rounded to fp32
    good = x @ q4.dequantize(a["Wq"], a["scale_bias"], N, K).T
    assert oracle.max_normalized_error(good.astype(np.float32), y, D, wl.EPI_NONE) <= oracle.TOL_F32_OUT
