"""GPU parity of the fused RMSNorm + rotary + cache write against the oracle.

Operation: "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
vllm/model_executor/models/deepseek_v2.py (kv_a_layernorm = RMSNorm;
rotary_emb = get_rope(..., is_neox_style=False)) and the MLA common forward
(q_pe and k_pe rotated by position, then concat_and_cache_mla).

Bar.  The GPU computes in fp32 and the oracle in fp64, each rounding once to
bf16, so a bf16 result may land on the neighbouring value:
|gpu - ref| <= 2^-7 |ref| for the normalised latent, plus 2^-20 (|a| + |b|)
for a rotated pair (a, b) (fp32 cancellation).  The fp8 cache quantises
those bf16 values, so its codes are equal or adjacent.  Everything not
written (padded slots, skipped tokens, the rest of the pool) is compared
byte for byte, and skipped tokens are counted exactly.
"""
import numpy as np
import pytest
import torch

import mla_paged_kv_concat_gb300 as mla
import oracle
from mla_paged_kv_concat_gb300 import workloads as W

from _helpers import Dev, assert_close, oracle_decode

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _check_bf16(got_bits, ref_bits, extra=0.0, what=""):
    g = oracle.bf16_value(got_bits)
    r = oracle.bf16_value(ref_bits)
    bound = 2.0 ** -7 * np.abs(r) + extra
    bad = ~(np.abs(g - r) <= bound)
    assert not bad.any(), (what, np.argwhere(bad)[:5].tolist(), g[bad][:5], r[bad][:5])


def _pair_mag(bits):
    v = np.abs(oracle.bf16_value(bits))
    m = v[..., 0::2] + v[..., 1::2]
    return np.repeat(m, 2, axis=-1)


def _run(w, x, *, fp8, q_pe_view=False, nbad=0):
    d = Dev(w)
    gamma = x.gamma.cuda()
    pos = torch.from_numpy(x.positions).cuda()
    table = torch.from_numpy(x.table).cuda()
    if q_pe_view:
        q = d.q.clone()
        q_pe = q[:, :, w.kv_lora_rank:]
    else:
        q = None
        q_pe = x.q_pe.cuda()
    mla.norm_rope_cache_write(d.kv_c, d.k_pe, d.cache, d.slot_mapping, gamma, x.eps, pos, table,
                              q_pe=q_pe, scale=d.kv_scale if fp8 else None, err_count=d.err)
    torch.cuda.synchronize()
    cache_ref = w.kv_cache.copy()
    q_ref = _bits(w.q[:, :, w.kv_lora_rank:] if q_pe_view else x.q_pe).copy()
    nslot, npos = oracle.norm_rope_cache_write(
        w.kv_c, w.k_pe, x.gamma, x.eps, x.positions, x.table, w.slot_mapping, cache_ref,
        block_size=w.block_size, kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim,
        kv_is_fp8=fp8, scale=w.kv_scale, q_pe=q_ref)
    assert npos == nbad
    assert int(d.err.item()) == nslot + npos
    return d, cache_ref, q_pe, q_ref


def _compare_cache(w, x, d, cache_ref, fp8):
    R, D = w.kv_lora_rank, w.head_dim
    got = d.cache_numpy().reshape(-1, D)
    ref = cache_ref.reshape(-1, D)
    ok_pos = (x.positions >= 0) & (x.positions < x.table.shape[0])
    rows = np.array([s for t, s in enumerate(w.slot_mapping) if s >= 0 and ok_pos[t]], np.int64)
    toks = np.array([t for t, s in enumerate(w.slot_mapping) if s >= 0 and ok_pos[t]], np.int64)
    others = np.setdiff1d(np.arange(ref.shape[0]), rows)
    assert got[others].tobytes() == ref[others].tobytes(), "rows not written must not change"
    if rows.size == 0:
        return
    if fp8:
        # sign-magnitude order of the codes: equal or adjacent
        def order(c):
            c = c.astype(np.int32)
            return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)
        diff = np.abs(order(got[rows]) - order(ref[rows]))
        assert diff.max() <= 1, np.argwhere(diff > 1)[:5].tolist()
        assert (diff == 0).mean() > 0.99
        return
    _check_bf16(got[rows, :R], ref[rows, :R], what="normed kv_c")
    k_pe_in = _bits(w.k_pe)[toks]
    _check_bf16(got[rows, R:], ref[rows, R:], 2.0 ** -20 * _pair_mag(k_pe_in), what="rotated k_pe")


@pytest.mark.parametrize("name,kw,fp8,nbad", [
    ("tiny", None, False, 1),
    ("per_shard", None, False, 0),
    ("nr_r256", dict(seq_lens=[150, 33, 700, 1], num_heads=32, kv_lora_rank=256,
                     write="random", num_write_tokens=300), False, 3),
    ("nr_fp8", dict(seq_lens=[150, 33, 700], num_heads=32, kv_lora_rank=256, kv_fp8=True,
                    kv_scale=0.05, write="all"), True, 2),
    ("nr_fp8_512", dict(seq_lens=[90, 200], num_heads=16, kv_fp8=True, kv_scale=0.3,
                        write="all"), True, 0),
])
def test_fused_write_matches_oracle(cuda_dev, name, kw, fp8, nbad):
    w = W.make(name) if kw is None else W.make_workload(name, seed=81, **kw)
    x = W.norm_rope_inputs(w, seed=5, num_bad_positions=nbad, table_scale=1.0)
    d, cache_ref, q_pe, q_ref = _run(w, x, fp8=fp8, nbad=nbad)
    _compare_cache(w, x, d, cache_ref, fp8)
    q_in = _bits(x.q_pe)
    _check_bf16(_bits(q_pe), q_ref, 2.0 ** -20 * _pair_mag(q_in), what="rotated q_pe")
    bad = (x.positions < 0) | (x.positions >= x.table.shape[0])
    assert np.array_equal(_bits(q_pe)[bad], q_in[bad])


def test_scaled_table_and_q_pe_as_rope_columns_of_q(cuda_dev):
    """A table with a magnitude factor (as the YaRN scale would give) and q_pe
    given as the rope columns of q (head stride R+P, row stride H(R+P))."""
    w = W.make_workload("nr_view", seed=82, seq_lens=[300, 1000, 77, 64], num_heads=16)
    x = W.norm_rope_inputs(w, seed=6, table_scale=1.25)
    d, cache_ref, q_pe, q_ref = _run(w, x, fp8=False, q_pe_view=True)
    _compare_cache(w, x, d, cache_ref, False)
    q_in = _bits(w.q[:, :, w.kv_lora_rank:])
    _check_bf16(_bits(q_pe), q_ref, 2.0 ** -20 * 1.25 * _pair_mag(q_in), what="q rope cols")


@pytest.mark.parametrize("H", [16, 128])
def test_fused_write_then_decode(cuda_dev, H):
    """The fused write feeding decode (rotated q rope columns, normalised and
    rotated cache rows), against the oracle doing the same two steps."""
    w = W.make_workload("nr_dec", seed=83 + H, seq_lens=[300, 1000, 77, 640], num_heads=H)
    x = W.norm_rope_inputs(w, seed=7)
    d = Dev(w)
    q = d.q.clone()
    mla.norm_rope_cache_write(d.kv_c, d.k_pe, d.cache, d.slot_mapping, x.gamma.cuda(), x.eps,
                              torch.from_numpy(x.positions).cuda(),
                              torch.from_numpy(x.table).cuda(), q_pe=q[:, :, w.kv_lora_rank:],
                              err_count=d.err)
    d.q = q
    o, lse = d.decode(mla.mla_num_kv_splits(w.max_seq_len, 148))
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    cache_ref = w.kv_cache.copy()
    q_ref = _bits(w.q).copy()
    oracle.norm_rope_cache_write(
        w.kv_c, w.k_pe, x.gamma, x.eps, x.positions, x.table, w.slot_mapping, cache_ref,
        block_size=w.block_size, kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim,
        kv_is_fp8=False, q_pe=q_ref[:, :, w.kv_lora_rank:])
    w.q = W.bits_to_torch_bf16(q_ref)
    o_ref, lse_ref = oracle_decode(w, cache_ref)
    assert_close(o, lse, o_ref, lse_ref, what=f"fused write + decode H={H}")
