"""GPU parity of the E5M2 cache: the write (plain and fused) and the decode
reading it, against the oracle's E5M2 codec.

Operation: "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
csrc/cache_kernels.cu (concat_and_cache_mla dispatched on kv_cache_dtype,
fp8 flavours E4M3 and E5M2) and vllm/attention/ops/triton_decode_attention.py
(decode over the dequantised cache).

Bar: the plain write is byte-exact (every finite bf16 value, several
scales); the decode meets |o - ref| <= 1e-2 + 1e-2 |ref|, |lse - ref| <= 2e-3;
the fused write's codes are equal or adjacent to the oracle's (its bf16
intermediate may round to the neighbouring value, see the fused-write tests).
"""
import numpy as np
import pytest
import torch

import mla_paged_kv_concat_gb300 as mla
import oracle
from mla_paged_kv_concat_gb300 import workloads as W

from _helpers import Dev, assert_close, sm_count

pytestmark = pytest.mark.gpu

E5 = "fp8_e5m2"


def _oracle_cache(w):
    cache = w.kv_cache.copy()
    oracle.cache_write(w.kv_c, w.k_pe, w.slot_mapping, cache, block_size=w.block_size,
                       kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim, kv_is_fp8=True,
                       scale=w.kv_scale, fp8_format="e5m2")
    return cache


def _write(d):
    mla.cache_write(d.kv_c, d.k_pe, d.cache, d.slot_mapping, kv_cache_dtype=E5,
                    scale=d.kv_scale, err_count=d.err)


@pytest.mark.parametrize("scale", [1.0, 0.05, 3.0, 1e-30, 3e37, 2.0 ** -130, 2.0 ** 127])
def test_e5m2_every_bf16_value(cuda_dev, scale):
    R, P = 256, 64
    D = R + P
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = W.bits_to_torch_bf16(bits).float().numpy()
    bits = bits[np.isfinite(vals)]
    T = (bits.size + D - 1) // D
    rows = np.concatenate([bits, np.zeros(T * D - bits.size, np.uint16)]).reshape(T, D)
    full = W.bits_to_torch_bf16(rows)
    bs = 64
    nb = (T + bs - 1) // bs
    w = W.make_workload("e5all", seed=55, seq_lens=[1], num_heads=1, kv_lora_rank=R,
                        pool_blocks=nb, block_size=bs, write="random", num_write_tokens=T)
    w.kv_c, w.k_pe = full[:, :R], full[:, R:]
    w.slot_mapping = np.arange(T, dtype=np.int64)
    w.kv_fp8, w.kv_scale = True, float(np.float32(scale))
    w.kv_cache = np.zeros((nb, bs, D), np.uint8)
    d = Dev(w)
    _write(d)
    torch.cuda.synchronize()
    assert d.cache_numpy().tobytes() == _oracle_cache(w).tobytes()


@pytest.mark.parametrize("R,H,splits", [(256, 32, 1), (256, 32, 8), (512, 16, 4),
                                        (512, 128, 4), (256, 3, 2)])
def test_e5m2_decode(cuda_dev, R, H, splits):
    w = W.make_workload("e5dec", seed=57 + H, seq_lens=[150, 33, 700, 1], num_heads=H,
                        kv_lora_rank=R, kv_fp8=True, kv_scale=0.05, write="all")
    d = Dev(w)
    _write(d)
    o, lse = mla.decode(d.q, d.cache, d.block_table, d.seq_lens, w.sm_scale, splits,
                        kv_lora_rank=R, kv_cache_dtype=E5, kv_scale=d.kv_scale,
                        err_count=d.err)
    torch.cuda.synchronize()
    cache = _oracle_cache(w)
    assert d.cache_numpy().tobytes() == cache.tobytes()
    o_ref, lse_ref = oracle.decode(w.q, cache, w.block_table, w.seq_lens,
                                   block_size=w.block_size, kv_lora_rank=R, rope_dim=w.rope_dim,
                                   sm_scale=w.sm_scale, kv_is_fp8=True, kv_scale=w.kv_scale,
                                   fp8_format="e5m2")
    assert_close(o, lse, o_ref, lse_ref, what=f"e5m2 R={R} H={H} S={splits}")
    # the same bytes read as E4M3 give another result: the format really is used
    o4, _ = mla.decode(d.q, d.cache, d.block_table, d.seq_lens, w.sm_scale, splits,
                       kv_lora_rank=R, kv_cache_dtype="fp8_e4m3", kv_scale=d.kv_scale)
    assert not torch.equal(o4, o)


def test_e5m2_fused_write(cuda_dev):
    w = W.make_workload("e5nr", seed=58, seq_lens=[150, 33, 700], num_heads=16,
                        kv_lora_rank=512, kv_fp8=True, kv_scale=0.3, write="all")
    x = W.norm_rope_inputs(w, seed=4, num_bad_positions=2)
    d = Dev(w)
    mla.norm_rope_cache_write(d.kv_c, d.k_pe, d.cache, d.slot_mapping, x.gamma.cuda(), x.eps,
                              torch.from_numpy(x.positions).cuda(),
                              torch.from_numpy(x.table).cuda(), kv_cache_dtype=E5,
                              scale=d.kv_scale, err_count=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 2
    ref = w.kv_cache.copy()
    oracle.norm_rope_cache_write(w.kv_c, w.k_pe, x.gamma, x.eps, x.positions, x.table,
                                 w.slot_mapping, ref, block_size=w.block_size,
                                 kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim,
                                 kv_is_fp8=True, scale=w.kv_scale, fp8_format="e5m2")
    got = d.cache_numpy().astype(np.int32)
    ref = ref.astype(np.int32)
    order = lambda c: np.where(c & 0x80, -(c & 0x7F), c & 0x7F)  # noqa: E731
    nan = (ref & 0x7F) > 0x7C
    assert np.array_equal(nan, (got & 0x7F) > 0x7C)
    diff = np.abs(order(got) - order(ref))[~nan]
    assert diff.max() <= 1 and (diff == 0).mean() > 0.99
