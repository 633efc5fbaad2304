"""Pins of the block-scaled (MX) oracle, oracle/mx.py, each against something
other than the oracle itself (CPU only).

* Decoders: every FP4 E2M1 code and selected E8M0 scale codes against the
  values the OCP Microscaling Formats (MX) Specification v1.0 defines
  (tests/golden/mx_formats.txt).
* mx_reference: exact rational brute force (fractions, with a decoder written
  here from the bit fields) on small problems of both element types; the
  special case of unit scales, which must equal the dense oracle on the same
  E4M3 bytes; the invariance under moving a power of two between a block's
  scale and its elements; and planted mistakes (block of 16, A's scales used
  for B, nibble order swapped, scale exponent off by one) all caught.
* The MX quantiser of the input generators: each element is the nearest
  representable value of x / X (ties to even) by brute force over the value
  table, and each block's largest element lands in the top binade.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from conftest import read_golden
from oracle import mx


# ------------------------------------------------------------------ decoders --

@pytest.mark.parametrize("row", read_golden("mx_formats.txt"), ids=lambda r: f"{r[0]}-{r[1]}")
def test_mx_decoders_match_the_specification(row):
    fmt, code, want = row[0], int(row[1], 16), float(row[2])
    got = float((mx.decode_e2m1 if fmt == "e2m1" else mx.decode_e8m0)(np.array([code]))[0])
    if np.isnan(want):
        assert np.isnan(got)
    else:
        assert got == want and np.signbit(got) == np.signbit(want)


def test_e2m1_decoder_covers_every_code_once():
    v = mx.decode_e2m1(np.arange(16))
    assert sorted(set(np.abs(v).tolist())) == list(wl.E2M1_MAGNITUDES)
    assert np.all(np.isfinite(v))


# ----------------------------------------------------- brute force (fractions) --

def _frac_e4m3(c):
    """E4M3 code -> Fraction, from the OFP8 bit fields (bias 7, 3 fraction bits)."""
    s, e, m = (c >> 7) & 1, (c >> 3) & 0xF, c & 7
    v = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -v if s else v


def _frac_e2m1(c):
    """E2M1 code -> Fraction, from the MX bit fields (bias 1, 1 fraction bit)."""
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    v = Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
    return -v if s else v


def _brute(M, N, K, elem, A, SA, B, SB, alpha, block=32, swap_nibbles_a=False, scales_b_from_a=False,
           scale_shift=0):
    """sum_k X^A a X^B b as exact fractions, with the storage read element by element."""
    def elem_at(codes, r, k, ld, swap=False):
        if elem == mx.ELEM_E4M3:
            return _frac_e4m3(int(codes[r * ld + k]))
        byte = int(codes[r * (ld // 2) + k // 2])
        odd = (k % 2 == 1) != swap
        return _frac_e2m1((byte >> 4) & 0xF if odd else byte & 0xF)

    def scale_at(codes, r, k):
        nb = K // block
        return Fraction(2) ** (int(codes[r * nb + k // block]) - 127 + scale_shift)

    out = np.zeros((M, N), dtype=object)
    for i in range(M):
        for j in range(N):
            acc = Fraction(0)
            for k in range(K):
                sb_codes, sb_row = (SA, i) if scales_b_from_a else (SB, j)
                acc += (scale_at(SA, i, k) * elem_at(A, i, k, K, swap_nibbles_a)) * \
                    (scale_at(sb_codes, sb_row, k) * elem_at(B, j, k, K))
            out[i, j] = Fraction(alpha) * acc
    return out


def _random_mx(seed, M, N, K, elem, scale_lo=124, scale_hi=131):
    g = torch.Generator().manual_seed(seed)
    if elem == mx.ELEM_E4M3:
        A = torch.randint(0, 256, (M * K,), generator=g)
        B = torch.randint(0, 256, (N * K,), generator=g)
        A = torch.where((A & 0x7F) == 0x7F, A - 1, A)        # no NaN codes
        B = torch.where((B & 0x7F) == 0x7F, B - 1, B)
    else:
        A = torch.randint(0, 256, (M * K // 2,), generator=g)
        B = torch.randint(0, 256, (N * K // 2,), generator=g)
    SA = torch.randint(scale_lo, scale_hi, (M * K // 32,), generator=g)
    SB = torch.randint(scale_lo, scale_hi, (N * K // 32,), generator=g)
    return [t.to(torch.uint8).numpy() for t in (A, SA, B, SB)]


def _ref(M, N, K, elem, A, SA, B, SB, alpha=1.0):
    y, D = mx.mx_reference(M, N, K, elem, A, K, SA, B, K, SB, None, N, wl.F32, alpha, 0.0, None, wl.EPI_NONE)
    return y, D


@pytest.mark.parametrize("elem", [mx.ELEM_E4M3, mx.ELEM_E2M1])
@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (2, 3, 64), (3, 2, 96)])
def test_mx_reference_against_rational_brute_force(elem, M, N, K):
    A, SA, B, SB = _random_mx(7 + M + N + K, M, N, K, elem)
    y, D = _ref(M, N, K, elem, A, SA, B, SB, alpha=1.5)
    want = _brute(M, N, K, elem, A, SA, B, SB, 1.5)
    for i in range(M):
        for j in range(N):
            # the float64 matmul rounds; its error is far below 2^-45 of the absolute sum
            assert abs(Fraction(y[i, j]) - want[i, j]) <= Fraction(D[i, j]) * Fraction(2) ** -45


@pytest.mark.parametrize("mistake", ["block_16", "b_scales_from_a", "nibbles_swapped", "scale_off_by_one"])
def test_planted_mistakes_fail_the_brute_force(mistake):
    """A reference with any of these mistakes differs from the oracle on random inputs
    by far more than rounding: the brute-force pin would catch each in the oracle.  (The
    nibble order is swapped in A alone: swapped in both operands it only permutes the sum
    within a block, which no product can see; test_e2m1_element_order pins it directly.)"""
    elem = mx.ELEM_E2M1 if mistake == "nibbles_swapped" else mx.ELEM_E4M3
    M, N, K = 2, 2, 64
    A, SA, B, SB = _random_mx(41, M, N, K, elem, scale_lo=120, scale_hi=134)
    y, D = _ref(M, N, K, elem, A, SA, B, SB)
    kw = {"block_16": dict(block=16), "b_scales_from_a": dict(scales_b_from_a=True),
          "nibbles_swapped": dict(swap_nibbles_a=True), "scale_off_by_one": dict(scale_shift=1)}[mistake]
    if mistake == "block_16":
        # block 16 reads K/16 scales per row: give it a scale array that long, first half the true one
        SA16 = np.concatenate([SA.reshape(M, -1), SA.reshape(M, -1)], axis=1).reshape(-1)
        SB16 = np.concatenate([SB.reshape(N, -1), SB.reshape(N, -1)], axis=1).reshape(-1)
        wrong = _brute(M, N, K, elem, A, SA16, B, SB16, 1.0, **kw)
    else:
        wrong = _brute(M, N, K, elem, A, SA, B, SB, 1.0, **kw)
    diff = max(abs(Fraction(y[i, j]) - wrong[i, j]) / max(Fraction(D[i, j]), Fraction(1, 2 ** 60))
               for i in range(M) for j in range(N))
    assert diff > Fraction(1, 1000)


# ---------------------------------------------- special cases and invariances --

def test_unit_scales_reduce_to_the_dense_oracle():
    """All scale codes 127 (X = 1): the MX product of E4M3 elements is the dense product of
    the same E4M3 bytes, B^T given as N x K (b_stride_k = 1, b_stride_n = K)."""
    M, N, K = 5, 6, 96
    A, _, B, _ = _random_mx(3, M, N, K, mx.ELEM_E4M3)
    SA = np.full(M * K // 32, 127, np.uint8)
    SB = np.full(N * K // 32, 127, np.uint8)
    bias = np.linspace(-1, 1, N).astype(np.float32)
    C = np.zeros(M * N, np.int32)
    y, D = mx.mx_reference(M, N, K, mx.ELEM_E4M3, A, K, SA, B, K, SB, C, N, wl.F32, 0.75, 0.0, bias,
                           wl.EPI_BIAS_GELU)
    y2, D2 = oracle.gemm_reference(M, N, K, wl.E4M3, A, K, 1, B, 1, K, C, N, wl.F32, 0.75, 0.0, bias,
                                   wl.EPI_BIAS_GELU)
    assert np.allclose(y, y2, rtol=1e-14, atol=1e-14 * float(D.max())) and np.allclose(D, D2, rtol=1e-14)


def test_power_of_two_moves_between_scale_and_elements():
    """Raising one block's scale code by one equals doubling that block's elements (E4M3
    codes whose exponent field is below 14 double exactly when it is raised by one)."""
    M, N, K = 2, 3, 64
    g = torch.Generator().manual_seed(9)
    e = torch.randint(1, 14, (M * K,), generator=g)
    m = torch.randint(0, 8, (M * K,), generator=g)
    s = torch.randint(0, 2, (M * K,), generator=g)
    A = ((s << 7) | (e << 3) | m).to(torch.uint8).numpy()
    _, SA, B, SB = _random_mx(10, M, N, K, mx.ELEM_E4M3)
    y0, _ = _ref(M, N, K, mx.ELEM_E4M3, A, SA, B, SB)
    SA1 = SA.copy()
    SA1[1 * (K // 32) + 1] += 1                      # row 1, block 1
    A1 = A.copy().astype(np.int64)
    blk = slice(1 * K + 32, 1 * K + 64)
    A1[blk] = A1[blk] + (1 << 3)                     # same block: exponent field + 1
    y1, _ = _ref(M, N, K, mx.ELEM_E4M3, A, SA1, B, SB)
    y2, _ = _ref(M, N, K, mx.ELEM_E4M3, A1.astype(np.uint8), SA, B, SB)
    assert np.array_equal(y1, y2) and not np.array_equal(y0, y1)


def test_e2m1_element_order():
    """Byte 0x21 holds element k = 0 in its low nibble (code 1: 0.5) and k = 1 in its high
    nibble (code 2: 1.0); the next byte holds k = 2 and 3."""
    v = mx.element_values(np.array([0x21, 0xF7], np.uint8), 1, 4, 4, mx.ELEM_E2M1)
    assert v.tolist() == [[0.5, 1.0, 6.0, -6.0]]
    # a product by hand: A = (0.5, 1.0, 0...), B = (1.0, 2.0, 0...), unit scales: 0.5 + 2.0
    K = 32
    A = np.zeros(K // 2, np.uint8)
    A[0] = 0x21
    B = np.zeros(K // 2, np.uint8)
    B[0] = 0x42
    S = np.full(1, 127, np.uint8)
    y, D = _ref(1, 1, K, mx.ELEM_E2M1, A, S, B, S)
    assert y[0, 0] == 2.5 and D[0, 0] == 2.5


def test_beta_and_alpha_zero_conventions():
    """alpha == 0 leaves the operands unread (NaN scales harmless); beta == 0 leaves C unread."""
    M, N, K = 2, 2, 32
    nan_scales = np.full(M * K // 32, 0xFF, np.uint8)
    C = np.array([0x3F800000, 0x40000000, 0x7FC00000, 0xBF800000], np.uint32).astype(np.int64)
    y, D = mx.mx_reference(M, N, K, mx.ELEM_E4M3, np.zeros(M * K, np.uint8), K, nan_scales,
                           np.zeros(N * K, np.uint8), K, nan_scales, C, N, wl.F32, 0.0, 2.0, None, wl.EPI_NONE)
    assert np.isnan(y[1, 0]) and y[0, 0] == 2.0 and y[0, 1] == 4.0 and y[1, 1] == -2.0
    A, SA, B, SB = _random_mx(5, M, N, K, mx.ELEM_E4M3)
    y, _ = mx.mx_reference(M, N, K, mx.ELEM_E4M3, A, K, SA, B, K, SB, C, N, wl.F32, 1.0, 0.0, None,
                           wl.EPI_NONE)
    assert np.all(np.isfinite(y))


# --------------------------------------------------------- the input quantiser --

def _value_table(elem):
    if elem == wl.MX_E4M3:
        t = oracle.decode_e4m3(np.arange(256))
    else:
        t = mx.decode_e2m1(np.arange(16))
    return np.unique(np.abs(t[np.isfinite(t)]))


@pytest.mark.parametrize("elem", [wl.MX_E4M3, wl.MX_E2M1])
def test_quantiser_rounds_to_nearest_even_in_the_top_binade(elem):
    x = wl.normal(12, 6, 128) * torch.tensor([1e-3, 1.0, 30.0, 1e4, 0.2, 7.0]).reshape(6, 1)
    x[5, 32:64] = 0.0                                   # an all-zero block
    codes, scales = wl.mx_quantize(x, elem)
    P = mx.element_values(codes.reshape(-1).numpy(), 6, 128, 128, elem)
    X = mx.block_scales(scales.reshape(-1).numpy(), 6, 128)
    table = _value_table(elem)
    emax = wl.MX_EMAX[elem]
    xv = x.to(torch.float64).numpy()
    for r in range(6):
        for b in range(4):
            blk = slice(32 * b, 32 * b + 32)
            amax = np.abs(xv[r, blk]).max()
            if amax == 0:
                assert np.all(P[r, blk] == 0)
                continue
            # the block's largest |x| / X lies in [2^emax, 2^(emax+1))
            top = amax / X[r, 32 * b]
            assert 2.0 ** emax <= top < 2.0 ** (emax + 1)
            for k in range(32 * b, 32 * b + 32):
                q = abs(xv[r, k] / X[r, k])
                q = min(q, table[-1])                   # saturation
                d = np.abs(table - q)
                best = table[d == d.min()]
                got = abs(P[r, k])
                assert got in best
                if best.size == 2:                      # a tie: the even code
                    codes_of = {float(v): c for c, v in enumerate(
                        (oracle.decode_e4m3(np.arange(128)) if elem == wl.MX_E4M3 else mx.decode_e2m1(np.arange(8))))}
                    assert codes_of[got] % 2 == 0
                assert np.sign(P[r, k]) in (np.sign(xv[r, k]), 0.0)
