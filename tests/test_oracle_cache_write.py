"""Pins for the oracle's cache write.

What it restates: "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
csrc/cache_kernels.cu, concat_and_cache_mla_kernel and its host wrapper
concat_and_cache_mla: token t with slot s >= 0 lands in block s / bs, row
s % bs, elements [0, R) from kv_c[t] and [R, R+P) from k_pe[t]; slot -1 is a
padded token.  Pinned here against numpy fancy-index assignment, which shares
nothing with the oracle's loop.
"""
import numpy as np
import pytest
import torch

from mla_paged_kv_concat_gb300 import workloads as W


def _setup(seed, T, R, P, NB, bs, fp8):
    rng = np.random.default_rng(seed)
    D = R + P
    cache = np.full((NB, bs, D), W.FP8_NAN if fp8 else W.BF16_NAN,
                    np.uint8 if fp8 else np.uint16)
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int64)
    kv_c = W.bits_to_torch_bf16(W.randn_bf16(rng, (T, R)))
    k_pe = W.bits_to_torch_bf16(W.randn_bf16(rng, (T, P)))
    return cache, slots, kv_c, k_pe


def _numpy_write(cache, slots, kv_c, k_pe, fp8, scale):
    """Reference: one fancy-index assignment of the concatenated rows."""
    rows = torch.cat([kv_c, k_pe], dim=1)
    if fp8:
        y = (rows.to(torch.float32).numpy() / np.float32(scale)).astype(np.float32)
        y = np.clip(y, -448.0, 448.0)  # satfinite; torch's cast does not saturate
        vals = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    else:
        vals = rows.view(torch.int16).numpy().view(np.uint16)
    keep = slots >= 0
    flat = cache.reshape(-1, cache.shape[-1])
    flat[slots[keep]] = vals[keep]


@pytest.mark.parametrize("R,fp8", [(512, False), (256, False), (512, True), (256, True)])
@pytest.mark.parametrize("bs", [16, 64])
def test_cache_write_equals_fancy_index(oracle_mod, R, fp8, bs):
    P, NB, T = 64, 9, 50
    cache, slots, kv_c, k_pe = _setup(7 + R + bs, T, R, P, NB, bs, fp8)
    slots[3] = -1
    slots[17] = -1
    ref = cache.copy()
    _numpy_write(ref, slots, kv_c, k_pe, fp8, 0.05)
    got = cache.copy()
    bad = oracle_mod.cache_write(kv_c, k_pe, slots, got, block_size=bs, kv_lora_rank=R,
                                 rope_dim=P, kv_is_fp8=fp8, scale=0.05)
    assert bad == 0
    assert np.array_equal(got, ref)


def test_cache_write_strided_views(oracle_mod):
    """kv_c and k_pe as column slices of one [T, R+P] projection output."""
    R, P, NB, bs, T = 512, 64, 4, 64, 20
    rng = np.random.default_rng(3)
    full = W.bits_to_torch_bf16(W.randn_bf16(rng, (T, R + P + 8)))
    kv_c, k_pe = full[:, :R], full[:, R:R + P]
    cache = np.zeros((NB, bs, R + P), np.uint16)
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int64)
    ref = cache.copy()
    _numpy_write(ref, slots, kv_c.contiguous(), k_pe.contiguous(), False, 1.0)
    oracle_mod.cache_write(kv_c, k_pe, slots, cache, block_size=bs, kv_lora_rank=R,
                           rope_dim=P, kv_is_fp8=False)
    assert np.array_equal(cache, ref)


@pytest.mark.parametrize("fp8", [False, True])
def test_padded_slot_leaves_cache_identical(oracle_mod, fp8):
    R, P, NB, bs = 512, 64, 3, 64
    cache, _, kv_c, k_pe = _setup(11, 5, R, P, NB, bs, fp8)
    before = cache.copy()
    bad = oracle_mod.cache_write(kv_c, k_pe, np.full(5, -1, np.int64), cache, block_size=bs,
                                 kv_lora_rank=R, rope_dim=P, kv_is_fp8=fp8, scale=0.05)
    assert bad == 0
    assert cache.tobytes() == before.tobytes()


def test_out_of_range_slot_skipped_and_counted(oracle_mod):
    R, P, NB, bs = 256, 64, 2, 16
    cache, _, kv_c, k_pe = _setup(12, 3, R, P, NB, bs, False)
    slots = np.array([NB * bs, 5, NB * bs + 100], np.int64)
    ref = cache.copy()
    _numpy_write(ref, np.array([-1, 5, -1], np.int64), kv_c, k_pe, False, 1.0)
    bad = oracle_mod.cache_write(kv_c, k_pe, slots, cache, block_size=bs, kv_lora_rank=R,
                                 rope_dim=P, kv_is_fp8=False)
    assert bad == 2
    assert np.array_equal(cache, ref)


def test_padded_block_stride(oracle_mod):
    """A block stride larger than bs * D leaves the gap between blocks alone."""
    R, P, NB, bs, T = 256, 64, 3, 16, 12
    D = R + P
    stride = bs * D + 64
    rng = np.random.default_rng(5)
    buf = np.full((NB, stride), 0x1234, np.uint16)
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int64)
    kv_c = W.bits_to_torch_bf16(W.randn_bf16(rng, (T, R)))
    k_pe = W.bits_to_torch_bf16(W.randn_bf16(rng, (T, P)))
    oracle_mod.cache_write(kv_c, k_pe, slots, buf, block_size=bs, kv_lora_rank=R, rope_dim=P,
                           kv_is_fp8=False, block_stride=stride)
    assert np.all(buf[:, bs * D:] == 0x1234)
    ref = np.full((NB, bs, D), 0x1234, np.uint16)
    _numpy_write(ref, slots, kv_c, k_pe, False, 1.0)
    assert np.array_equal(buf[:, :bs * D].reshape(NB, bs, D), ref)
