"""GPU parity of the cache write: byte-exact against the oracle, fp8 included.

Operation: "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
csrc/cache_kernels.cu, concat_and_cache_mla_kernel.
"""
import numpy as np
import pytest
import torch

import mla_paged_kv_concat_gb300 as mla
from mla_paged_kv_concat_gb300 import workloads as W

from _helpers import Dev, oracle_cache

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "per_shard", "fp8_small"])
def test_named_workload_write_is_byte_exact(cuda_dev, name):
    w = W.make(name)
    d = Dev(w)
    d.write()
    torch.cuda.synchronize()
    got = d.cache_numpy()
    ref = oracle_cache(w)
    assert got.tobytes() == ref.tobytes()
    assert int(d.err.item()) == 0


@pytest.mark.parametrize("R", [512, 256])
@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("bs", [1, 16, 64, 100])
def test_random_slots_all_layouts(cuda_dev, R, fp8, bs):
    nb = 11
    w = W.make_workload("cw", seed=40 + R + bs + fp8, seq_lens=[1], num_heads=1,
                        kv_lora_rank=R, pool_blocks=nb, block_size=bs, write="random",
                        num_write_tokens=min(37, nb * bs - 1), kv_fp8=False)
    w.kv_fp8 = fp8
    w.kv_scale = float(np.float32(0.05))
    w.kv_cache = np.full(w.kv_cache.shape, W.FP8_NAN if fp8 else W.BF16_NAN,
                         np.uint8 if fp8 else np.uint16)
    d = Dev(w)
    d.write()
    torch.cuda.synchronize()
    assert d.cache_numpy().tobytes() == oracle_cache(w).tobytes()


def test_fp8_edge_values(cuda_dev):
    """Saturation, ties, subnormals and NaN through the fp8 write."""
    scale = np.float32(0.05)
    edge = np.array([0.0, -0.0, 22.4, -22.4, 23.2, 1e6, -1e6, 448 * 0.05, 464 * 0.05,
                     2 ** -9 * 0.05, 2 ** -10 * 0.05, 1.0625 * 0.05, 3e38, -3e38],
                    np.float32)
    R, P, T = 512, 64, 4
    rng = np.random.default_rng(9)
    x = rng.standard_normal((T, R + P)).astype(np.float32) * 30
    x.flat[:edge.size] = edge
    x.flat[edge.size:edge.size + 3] = np.nan
    bits = W.bf16_bits_from_f32(x)
    bits.flat[edge.size:edge.size + 3] = [0x7FC0, 0xFFC0, 0x7F81]
    full = W.bits_to_torch_bf16(bits)
    w = W.make_workload("fp8e", seed=50, seq_lens=[1], num_heads=1, pool_blocks=2,
                        block_size=64, write="random", num_write_tokens=T)
    w.kv_c, w.k_pe = full[:, :R], full[:, R:]
    w.slot_mapping = np.array([0, 65, 3, 127], np.int64)
    w.kv_fp8, w.kv_scale = True, float(scale)
    w.kv_cache = np.zeros(w.kv_cache.shape, np.uint8)
    d = Dev(w)
    d.write()
    torch.cuda.synchronize()
    got, ref = d.cache_numpy(), oracle_cache(w)
    nan_in = np.isnan(full.float().numpy()).reshape(-1)
    # positions that received a NaN input: both sides must hold a NaN code
    flat_got = got.reshape(-1, R + P)
    flat_ref = ref.reshape(-1, R + P)
    rows = w.slot_mapping
    g, r = flat_got[rows].reshape(-1), flat_ref[rows].reshape(-1)
    assert np.all((g[nan_in] & 0x7F) == 0x7F) and np.all((r[nan_in] & 0x7F) == 0x7F)
    assert np.array_equal(g[~nan_in], r[~nan_in])
    other = np.ones(flat_got.shape[0], bool)
    other[rows] = False
    assert np.array_equal(flat_got[other], flat_ref[other])


def test_strided_and_unaligned_sources(cuda_dev):
    """kv_c/k_pe as column slices of one projection output; an odd column
    offset forces the element-wise path."""
    R, P, T, nb, bs = 512, 64, 20, 4, 64
    rng = np.random.default_rng(7)
    for off in (0, 1):
        full = W.bits_to_torch_bf16(W.randn_bf16(rng, (T, R + P + 9)))
        w = W.make_workload("strided", seed=51, seq_lens=[1], num_heads=1, pool_blocks=nb,
                            write="random", num_write_tokens=T)
        w.kv_c, w.k_pe = full[:, off:off + R], full[:, off + R:off + R + P]
        d = Dev(w)
        d.kv_c = full.cuda()[:, off:off + R]
        d.k_pe = full.cuda()[:, off + R:off + R + P]
        d.write()
        torch.cuda.synchronize()
        assert d.cache_numpy().tobytes() == oracle_cache(w).tobytes()


def test_padded_slots_and_out_of_range(cuda_dev):
    w = W.make_workload("oor", seed=52, seq_lens=[1], num_heads=1, pool_blocks=3,
                        write="random", num_write_tokens=6)
    w.slot_mapping = np.array([-1, 3 * 64, 5, -1, 3 * 64 + 1000, 70], np.int64)
    d = Dev(w)
    before = d.cache_numpy().copy()
    d.write()
    torch.cuda.synchronize()
    got = d.cache_numpy()
    assert got.tobytes() == oracle_cache(w).tobytes()
    assert int(d.err.item()) == 2
    changed = np.nonzero((got != before).any(axis=2).reshape(-1))[0]
    assert set(changed.tolist()) <= {5, 70}


def test_num_tokens_smaller_than_rows(cuda_dev):
    """slot_mapping shorter than kv_c (CUDA-graph padding of the inputs)."""
    w = W.make_workload("pad", seed=53, seq_lens=[1], num_heads=1, pool_blocks=2,
                        write="random", num_write_tokens=8)
    d = Dev(w)
    d.slot_mapping = d.slot_mapping[:5]
    w.slot_mapping = w.slot_mapping[:5]
    d.write()
    torch.cuda.synchronize()
    assert d.cache_numpy().tobytes() == oracle_cache(w).tobytes()


@pytest.mark.parametrize("scale", [1.0, 0.05, 0.3, 7.0, 1e-30, 3e37, 2.0 ** -130, 2.0 ** 127])
def test_fp8_every_bf16_value(cuda_dev, scale):
    """Every finite bf16 bit pattern through the fp8 write, byte-exact against
    the oracle's IEEE division and E4M3 rounding (ties, subnormals, saturation,
    and quotients next to a rounding boundary, where the kernel falls back to
    the division)."""
    R, P = 256, 64
    D = R + P
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = W.bits_to_torch_bf16(bits).float().numpy()
    bits = bits[np.isfinite(vals)]
    T = (bits.size + D - 1) // D
    pad = np.zeros(T * D - bits.size, np.uint16)
    rows = np.concatenate([bits, pad]).reshape(T, D)
    full = W.bits_to_torch_bf16(rows)
    bs = 64
    nb = (T + bs - 1) // bs
    w = W.make_workload("fp8all", seed=54, seq_lens=[1], num_heads=1, kv_lora_rank=R,
                        pool_blocks=nb, block_size=bs, write="random", num_write_tokens=T)
    w.kv_c, w.k_pe = full[:, :R], full[:, R:]
    w.slot_mapping = np.arange(T, dtype=np.int64)
    w.kv_fp8, w.kv_scale = True, float(np.float32(scale))
    w.kv_cache = np.zeros((nb, bs, D), np.uint8)
    d = Dev(w)
    d.write()
    torch.cuda.synchronize()
    assert d.cache_numpy().tobytes() == oracle_cache(w).tobytes()
