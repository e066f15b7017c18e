"""Pins for the oracle's scalar codecs (bf16 value, E4M3 value and encode).

The E4M3 format is OCP 8-bit floating point "E4M3" (e4m3fn): bias 7, no
infinities, NaN = S.1111.111, max normal 448, min normal 2^-6, min subnormal
2^-9.  The pages only say "fp8" for the cache ("frozenleaves/vllm compare
v0.11.0...mla_cuda_graphs", csrc/cache_kernels.cu, concat_and_cache_mla_kernel
calls fp8::scaled_convert); the reading is this format with round to nearest
even and saturation of finite overflow.
"""
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def all_bf16_patterns():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def test_bf16_value_all_patterns(oracle_mod):
    bits = all_bf16_patterns()
    got = oracle_mod.bf16_value(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # sign of zero is kept
    assert np.signbit(oracle_mod.bf16_value(np.array([0x8000], np.uint16)))[0]


def test_e4m3_value_against_torch_all_codes(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle_mod.e4m3_value(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.nonzero(nan)[0], [0x7F, 0xFF])
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def _load_landmarks():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_landmarks.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                code, val = line.split()
                rows.append((int(code, 16), float(val)))
    return rows


def test_e4m3_value_landmarks(oracle_mod):
    rows = _load_landmarks()
    assert len(rows) >= 10
    for code, val in rows:
        got = oracle_mod.e4m3_value(np.array([code], np.uint8))[0]
        if np.isnan(val):
            assert np.isnan(got), hex(code)
        else:
            assert got == val and np.signbit(got) == np.signbit(val), (hex(code), got, val)


def test_e4m3_value_is_monotone_on_positive_codes(oracle_mod):
    v = oracle_mod.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(v) > 0)
    assert v[0x7E] == 448.0 and v[1] == 2.0 ** -9 and v[8] == 2.0 ** -6


@pytest.mark.parametrize("divide_by", [None, 0.05])
def test_e4m3_encode_matches_torch_cast_on_all_bf16(oracle_mod, divide_by):
    bits = all_bf16_patterns()
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    y = x if divide_by is None else (x / np.float32(divide_by)).astype(np.float32)
    keep = np.isfinite(y) & (np.abs(y) <= 448.0)
    y = y[keep]
    got = oracle_mod.e4m3_encode(y)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(y[i]), hex(got[i]), hex(ref[i])) for i in bad[:8]]


@pytest.mark.parametrize("y,code", [
    (0.0, 0x00), (-0.0, 0x80), (1.0, 0x38), (-1.0, 0xB8),
    (448.0, 0x7E), (-448.0, 0xFE),
    (464.0, 0x7E),            # tie between 448 and 480: 448 has the even mantissa
    (449.0, 0x7E), (1e30, 0x7E), (float("inf"), 0x7E), (float("-inf"), 0xFE),
    (2.0 ** -9, 0x01), (2.0 ** -10, 0x00),          # tie between 0 and 2^-9 -> 0
    (3 * 2.0 ** -10, 0x02),                          # tie between 1 and 2 (x 2^-9) -> 2
    (1.0625, 0x38), (1.1875, 0x3A),                  # mantissa ties -> even
    (1e-30, 0x00), (-1e-30, 0x80),
    (15 * 2.0 ** -10, 0x08),                         # 7.5 * 2^-9 rounds up to min normal
])
def test_e4m3_encode_edges(oracle_mod, y, code):
    got = oracle_mod.e4m3_encode(np.array([y], np.float32))[0]
    assert got == code, (y, hex(got), hex(code))


def test_e4m3_encode_nan(oracle_mod):
    got = oracle_mod.e4m3_encode(np.array([np.nan, -np.nan], np.float32))
    assert np.all(np.isnan(oracle_mod.e4m3_value(got)))


def test_e4m3_roundtrip_all_finite_codes(oracle_mod):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle_mod.e4m3_value(codes).astype(np.float32)
    assert np.array_equal(oracle_mod.e4m3_encode(vals), codes)
