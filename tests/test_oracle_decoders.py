"""Pins for the oracle's element decoders (CPU only).

Each decoder is checked (1) against the exact values the format definitions
fix for selected codes (golden fixture with its sources) and (2) exhaustively,
code by code, against PyTorch's CPU conversions, an implementation the oracle
does not use.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

FORMATS = {"f16": oracle.F16, "bf16": oracle.BF16, "f32": oracle.F32, "e4m3": oracle.E4M3}


def _same(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    eq = (a == b) & (np.signbit(a) == np.signbit(b))
    return both_nan | eq


@pytest.mark.parametrize("row", read_golden("number_formats.txt"), ids=lambda r: f"{r[0]}-{r[1]}")
def test_spec_values(row):
    fmt, code, value = row
    got = oracle.decode(np.array([int(code, 16)]), FORMATS[fmt])[0]
    want = float(value)
    assert _same(got, want), (fmt, code, got, want)


def test_f16_exhaustive_against_torch():
    codes = np.arange(1 << 16, dtype=np.int64)
    ref = torch.from_numpy(codes.astype(np.int32)).to(torch.int16).view(torch.float16).to(torch.float64).numpy()
    assert _same(oracle.decode_f16(codes), ref).all()


def test_bf16_exhaustive_against_torch():
    codes = np.arange(1 << 16, dtype=np.int64)
    ref = torch.from_numpy(codes.astype(np.int32)).to(torch.int16).view(torch.bfloat16).to(torch.float64).numpy()
    assert _same(oracle.decode_bf16(codes), ref).all()


def test_e4m3_exhaustive_against_torch():
    codes = np.arange(256, dtype=np.int64)
    ref = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert _same(oracle.decode_e4m3(codes), ref).all()
    finite = oracle.decode_e4m3(codes)
    finite = finite[np.isfinite(finite)]
    assert finite.max() == 448.0 and finite.min() == -448.0
    assert np.isnan(oracle.decode_e4m3(codes)).sum() == 2  # S.1111.111 for both signs


def test_f32_sampled_against_torch():
    rng = np.random.default_rng(0)
    codes = np.concatenate([rng.integers(0, 1 << 32, size=1 << 20, dtype=np.int64),
                            np.arange(0, 1 << 12), (1 << 32) - 1 - np.arange(0, 1 << 12),
                            np.array([0x7F800000, 0xFF800000, 0x00800000, 0x007FFFFF])])
    ref = torch.from_numpy(codes.astype(np.uint32).view(np.int32)).view(torch.float32).to(torch.float64).numpy()
    assert _same(oracle.decode_f32(codes), ref).all()


def test_e4m3_grid_is_the_ocp_grid():
    """Positive finite E4M3 values are m*2^-9 (m<8) and (8+m)*2^(e-10), strictly increasing."""
    vals = oracle.decode_e4m3(np.arange(0x7F))
    expect = [m * 2.0 ** -9 for m in range(8)] + [(8 + m) * 2.0 ** (e - 10) for e in range(1, 16)
                                                 for m in range(8)][:0x7F - 8]
    assert np.array_equal(vals, np.array(expect))
    assert np.all(np.diff(vals) > 0)


def test_fp32_value_rounds_like_binary32():
    assert oracle.fp32_value(0.1) == float(np.float32(0.1)) != 0.1
    assert oracle.fp32_value(1.5) == 1.5
    assert math.isinf(oracle.fp32_value(1e39))
