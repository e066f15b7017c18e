"""Pins for the oracle's E5M2 codec (the cache's second fp8 flavour).

The pages dispatch the cache write on a kv_cache_dtype string
("frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
csrc/cache_kernels.cu, concat_and_cache_mla: DISPATCH_BY_KV_CACHE_DTYPE),
whose fp8 flavours are E4M3 and E5M2.  E5M2 is the OCP 8-bit floating point
"E5M2" format: bias 15, IEEE-like infinities and NaNs, max normal 57344,
min normal 2^-14, min subnormal 2^-16.  The reading for the encode is the
one taken for E4M3: x / scale in fp32, round to nearest even, finite
overflow and infinities saturated to +-57344, NaN to a NaN code.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from mla_paged_kv_concat_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _landmarks():
    rows = []
    with open(os.path.join(GOLDEN, "e5m2_landmarks.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                code, val = line.split()
                rows.append((int(code, 16), float(val)))
    return rows


def test_e5m2_value_landmarks(oracle_mod):
    rows = _landmarks()
    assert len(rows) >= 12
    for code, val in rows:
        got = oracle.e5m2_value(np.array([code], np.uint8))[0]
        if np.isnan(val):
            assert np.isnan(got), hex(code)
        else:
            assert got == val and np.signbit(got) == np.signbit(val), (hex(code), got, val)


def test_e5m2_value_against_torch_all_codes(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e5m2_value(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("divide_by", [None, 0.05, 3.0])
def test_e5m2_encode_matches_torch_cast_on_all_bf16(oracle_mod, divide_by):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    y = x if divide_by is None else (x / np.float32(divide_by)).astype(np.float32)
    keep = np.isfinite(y) & (np.abs(y) <= 57344.0)
    y = y[keep]
    got = oracle.e5m2_encode(y)
    ref = torch.from_numpy(y).to(torch.float8_e5m2).view(torch.uint8).numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(y[i]), hex(got[i]), hex(ref[i])) for i in bad[:8]]


@pytest.mark.parametrize("y,code", [
    (0.0, 0x00), (-0.0, 0x80), (1.0, 0x3C), (-1.25, 0xBD),
    (57344.0, 0x7B), (-57344.0, 0xFB),
    (61440.0, 0x7B),            # the tie above max normal: saturates, not infinity
    (1e30, 0x7B), (float("inf"), 0x7B), (float("-inf"), 0xFB),
    (2.0 ** -16, 0x01), (2.0 ** -17, 0x00),          # tie between 0 and 2^-16 -> 0
    (3 * 2.0 ** -17, 0x02),                          # tie between 1 and 2 (x 2^-16) -> 2
    (1.125, 0x3C), (1.375, 0x3E),                    # mantissa ties -> even
    (7 * 2.0 ** -17, 0x04),                          # 3.5 * 2^-16 rounds up to min normal
])
def test_e5m2_encode_edges(oracle_mod, y, code):
    got = oracle.e5m2_encode(np.array([y], np.float32))[0]
    assert got == code, (y, hex(got), hex(code))


def test_e5m2_encode_nan_and_roundtrip(oracle_mod):
    assert np.all(np.isnan(oracle.e5m2_value(oracle.e5m2_encode(
        np.array([np.nan, -np.nan], np.float32)))))
    codes = np.array([c for c in range(256) if (c & 0x7F) < 0x7C], np.uint8)
    vals = oracle.e5m2_value(codes).astype(np.float32)
    assert np.array_equal(oracle.e5m2_encode(vals), codes)


def test_e5m2_cache_write_and_decode_use_the_e5m2_codec(oracle_mod):
    """The cache write stores E5M2(x / scale) and the decode reads
    E5M2 value * scale: checked against the codec on a small workload, and
    the decode against the same workload dequantised to fp64 by hand."""
    w = W.make_workload("e5m2", seed=71, seq_lens=[70, 3], num_heads=4, kv_lora_rank=256,
                        kv_fp8=True, kv_scale=0.3, write="all")
    cache = w.kv_cache.copy()
    oracle.cache_write(w.kv_c, w.k_pe, w.slot_mapping, cache, block_size=w.block_size,
                       kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim, kv_is_fp8=True,
                       scale=w.kv_scale, fp8_format="e5m2")
    D = w.head_dim
    kv = np.concatenate([w.kv_c.float().numpy(), w.k_pe.float().numpy()], axis=1)
    want = oracle.e5m2_encode((kv / np.float32(w.kv_scale)).astype(np.float32))
    flat = cache.reshape(-1, D)
    assert np.array_equal(flat[w.slot_mapping], want)
    o, lse = oracle.decode(w.q, cache, w.block_table, w.seq_lens, block_size=w.block_size,
                           kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim,
                           sm_scale=w.sm_scale, kv_is_fp8=True, kv_scale=w.kv_scale,
                           fp8_format="e5m2")
    # by hand: gather, dequantise, softmax, weighted sum (torch float64)
    q = torch.from_numpy(oracle.bf16_value(w.q.view(torch.int16).numpy().view(np.uint16)))
    for b, L in enumerate(w.seq_lens):
        toks = np.arange(int(L))
        slots = w.block_table[b, toks // w.block_size].astype(np.int64) * w.block_size \
            + toks % w.block_size
        K = torch.from_numpy(oracle.e5m2_value(flat[slots]) * w.kv_scale)
        s = (q[b] @ K.T) * w.sm_scale
        ref_o = torch.softmax(s, dim=-1) @ K[:, :w.kv_lora_rank]
        ref_l = torch.logsumexp(s, dim=-1)
        n = w.num_heads
        assert np.allclose(o[b * n:(b + 1) * n], ref_o.numpy(), rtol=1e-12, atol=1e-12)
        assert np.allclose(lse[b * n:(b + 1) * n], ref_l.numpy(), rtol=0, atol=1e-12)
