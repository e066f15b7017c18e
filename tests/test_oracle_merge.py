"""Pins for the oracle's cross-shard LSE merge.

What it restates: with decode context parallelism every rank attends over its
shard of the KV tokens and the (o, lse) pairs are combined by their
log-sum-exp ("Triton and MLA: portable attention and multi-head latent
attention", Design motivation: cp_lse_ag_out_rs; "vllm.v1.attention.backends.mla.
triton_mla", decode with DCP).  Pinned against the direct definition: the
decode of disjoint token shards, merged, equals the decode of the whole
sequence; and against the closed forms of the special cases.
"""
import numpy as np
import pytest

from mla_paged_kv_concat_gb300 import workloads as W

import oracle


def _shards(w, cuts):
    """Per shard: (block_table, seq_lens) of the token ranges [cuts[g], cuts[g+1])
    of every sequence (cuts [B, G+1], multiples of block_size)."""
    bs = w.block_size
    B, maxb = w.block_table.shape
    out = []
    for g in range(cuts.shape[1] - 1):
        bt = np.zeros_like(w.block_table)
        sl = np.zeros(B, np.int32)
        for b in range(B):
            a, z = int(cuts[b, g]), int(cuts[b, g + 1])
            n = (z - a + bs - 1) // bs
            bt[b, :n] = w.block_table[b, a // bs:a // bs + n]
            bt[b, n:] = w.block_table[b, -1]
            sl[b] = z - a
        out.append((bt, sl))
    return out


@pytest.mark.parametrize("G,seed", [(2, 1), (3, 2), (5, 3)])
def test_merged_shards_equal_direct_decode(oracle_mod, G, seed):
    w = W.make_workload("dcp", seed=70 + seed, seq_lens=[130, 257, 64, 700], num_heads=4)
    cache = w.kv_cache.copy()  # the batch's new tokens written, as decode sees it
    oracle.cache_write(w.kv_c, w.k_pe, w.slot_mapping, cache, block_size=w.block_size,
                       kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim, kv_is_fp8=False)
    rng = np.random.default_rng(seed)
    bs = w.block_size
    B = w.num_seqs
    cuts = np.zeros((B, G + 1), np.int64)
    for b, L in enumerate(w.seq_lens):
        pages = (int(L) + bs - 1) // bs
        inner = np.sort(rng.integers(0, pages + 1, size=G - 1)) * bs  # empty shards allowed
        cuts[b] = np.concatenate([[0], np.minimum(inner, L), [L]])
    kw = dict(block_size=bs, kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim,
              sm_scale=w.sm_scale)
    parts = [oracle.decode(w.q, cache, bt, sl, **kw) for bt, sl in _shards(w, cuts)]
    o_parts = np.stack([p[0] for p in parts])
    lse_parts = np.stack([p[1] for p in parts])
    o, lse = oracle.lse_merge(o_parts, lse_parts)
    o_ref, lse_ref = oracle.decode(w.q, cache, w.block_table, w.seq_lens, **kw)
    assert np.isfinite(o_ref).all()
    assert np.allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_special_cases(oracle_mod):
    R = 8
    rng = np.random.default_rng(4)
    a = rng.standard_normal((3, R))
    # every part empty
    o, lse = oracle.lse_merge(np.zeros((2, 1, R)), np.full((2, 1), -np.inf))
    assert np.all(o == 0) and lse[0] == -np.inf
    # one non-empty part: returned as it is
    o, lse = oracle.lse_merge(np.stack([a[:1], a[1:2]]), np.array([[-np.inf], [1.25]]))
    assert np.array_equal(o[0], a[1]) and lse[0] == 1.25
    # equal lse: the mean, and lse + ln G
    o, lse = oracle.lse_merge(a[:, None, :], np.full((3, 1), 0.5))
    assert np.allclose(o[0], a.mean(axis=0), rtol=0, atol=1e-15)
    assert abs(lse[0] - (0.5 + np.log(3))) < 1e-15
    # two parts, closed form
    l1, l2 = 0.3, -1.7
    o, lse = oracle.lse_merge(a[:2, None, :], np.array([[l1], [l2]]))
    w1, w2 = np.exp(l1), np.exp(l2)
    assert np.allclose(o[0], (w1 * a[0] + w2 * a[1]) / (w1 + w2), rtol=0, atol=1e-15)
    assert abs(lse[0] - np.log(w1 + w2)) < 1e-15
