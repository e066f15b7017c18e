"""Pins for the oracle's decode.

What it restates: MLA decode as MQA over the latent cache ("Triton and MLA:
portable attention and multi-head latent attention", Data flow: the cached row
is [kv_c | k_pe], fetched once MQA-style; V is the kv_c part), with scores
sm_scale * q.k over all R+P dims, softmax over the sequence, o = P.V and a
natural-log lse ("frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
vllm/attention/ops/triton_decode_attention.py, _fwd_grouped_kernel_stage1 and
_fwd_kernel_stage2).

Pinned against things that share nothing with the oracle's C loops:
torch CPU float64 scaled_dot_product_attention and logsumexp over K/V gathered
with numpy indexing; closed forms (L = 1 returns v exactly; equal scores give
the mean of v and lse = s + ln L); a math.fsum log-sum-exp; and the split-KV
route agreeing with the direct route.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from mla_paged_kv_concat_gb300 import workloads as W


def gather_kv(w, cache, b):
    """[L, D] float64 latent rows of sequence b, gathered with numpy indexing."""
    L = int(w.seq_lens[b])
    bs = w.block_size
    pages = w.block_table[b, :(L + bs - 1) // bs]
    rows = cache[pages].reshape(-1, cache.shape[-1])[:L]
    if w.kv_fp8:
        vals = torch.from_numpy(np.ascontiguousarray(rows)).view(torch.float8_e4m3fn)
        return vals.to(torch.float64) * float(np.float32(w.kv_scale))
    return torch.from_numpy(np.ascontiguousarray(rows).view(np.int16)).view(
        torch.bfloat16).to(torch.float64)


def sdpa_reference(w, cache):
    """torch float64 SDPA + logsumexp per row; returns o [rows*H, R], lse [rows*H]."""
    R = w.kv_lora_rank
    outs, lses = [], []
    qf = w.q.to(torch.float64)
    for r in range(w.num_rows):
        b = r // w.rows_per_seq
        K = gather_kv(w, cache, b)
        Q = qf[r]  # [H, D]
        if K.shape[0] == 0:
            outs.append(torch.zeros(w.num_heads, R, dtype=torch.float64))
            lses.append(torch.full((w.num_heads,), -math.inf, dtype=torch.float64))
            continue
        o = F.scaled_dot_product_attention(Q[:, None, :], K[None].expand(w.num_heads, -1, -1),
                                           K[None, :, :R].expand(w.num_heads, -1, -1),
                                           scale=w.sm_scale)[:, 0, :]
        lse = torch.logsumexp(w.sm_scale * (Q @ K.T), dim=-1)
        outs.append(o)
        lses.append(lse)
    return torch.cat(outs).numpy(), torch.cat(lses).numpy()


def written_cache(oracle_mod, w):
    cache = w.kv_cache.copy()
    oracle_mod.cache_write(w.kv_c, w.k_pe, w.slot_mapping, cache, block_size=w.block_size,
                           kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim,
                           kv_is_fp8=w.kv_fp8, scale=w.kv_scale)
    return cache


def oracle_decode(oracle_mod, w, cache, **kw):
    return oracle_mod.decode(w.q, cache, w.block_table, w.seq_lens, block_size=w.block_size,
                             kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim,
                             sm_scale=w.sm_scale, kv_is_fp8=w.kv_fp8, kv_scale=w.kv_scale, **kw)


CASES = [
    dict(seq_lens=[37, 130], num_heads=16),
    dict(seq_lens=[1, 64, 65, 300], num_heads=4, block_size=16),
    dict(seq_lens=[200, 7], num_heads=3, rows_per_seq=3),
    dict(seq_lens=[90, 129], num_heads=5, kv_lora_rank=256),
    dict(seq_lens=[150, 33], num_heads=4, kv_lora_rank=256, kv_fp8=True, kv_scale=0.05,
         write="all"),
    dict(seq_lens=[70], num_heads=2, kv_fp8=True, kv_scale=0.05, write="all", block_size=32),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_decode_matches_torch_sdpa_float64(oracle_mod, case):
    kw = dict(CASES[case])
    w = W.make_workload(f"case{case}", seed=100 + case, pool_blocks=None, **kw)
    cache = written_cache(oracle_mod, w)
    o, lse = oracle_decode(oracle_mod, w, cache)
    o_ref, lse_ref = sdpa_reference(w, cache)
    assert not np.isnan(o).any()
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


def test_named_tiny_workload_matches_sdpa_and_reads_no_poison(oracle_mod):
    w = W.make("tiny")
    cache = written_cache(oracle_mod, w)
    o, lse = oracle_decode(oracle_mod, w, cache)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    o_ref, lse_ref = sdpa_reference(w, cache)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fp8", [False, True])
def test_length_one_returns_v_exactly(oracle_mod, fp8):
    w = W.make_workload("l1", seed=21, seq_lens=[1, 1], num_heads=8, kv_fp8=fp8,
                        kv_scale=0.05, write="all" if fp8 else "newest")
    cache = written_cache(oracle_mod, w)
    o, lse = oracle_decode(oracle_mod, w, cache)
    for b in range(2):
        K = gather_kv(w, cache, b).numpy()
        v = K[0, :w.kv_lora_rank]
        qf = w.q.to(torch.float64).numpy()[b]
        for h in range(w.num_heads):
            assert np.array_equal(o[b * w.num_heads + h], v)
            s0 = w.sm_scale * math.fsum(qf[h] * K[0])
            assert abs(lse[b * w.num_heads + h] - s0) <= 1e-12 * max(1.0, abs(s0))


def test_equal_scores_give_mean_of_v(oracle_mod):
    """q is zero except its rope part and every token has the same k_pe, so all
    scores are equal: o = mean_j v_j and lse = s + ln L."""
    w = W.make_workload("eq", seed=22, seq_lens=[77, 200], num_heads=6)
    cache = written_cache(oracle_mod, w)
    R, D = w.kv_lora_rank, w.head_dim
    kpe = W.randn_bf16(np.random.default_rng(5), (D - R,))
    for b in range(2):
        L = int(w.seq_lens[b])
        for j in range(L):
            cache[w.block_table[b, j // 64], j % 64, R:] = kpe
    qb = w.q.view(torch.int16).numpy().view(np.uint16).copy()
    qb[:, :, :R] = 0
    w.q = W.bits_to_torch_bf16(qb)
    o, lse = oracle_decode(oracle_mod, w, cache)
    kpe_f = torch.from_numpy(kpe.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    qf = w.q.to(torch.float64).numpy()
    for b in range(2):
        L = int(w.seq_lens[b])
        V = gather_kv(w, cache, b).numpy()[:, :R]
        mean_v = np.array([math.fsum(V[:, d]) / L for d in range(R)])
        for h in range(w.num_heads):
            k = b * w.num_heads + h
            np.testing.assert_allclose(o[k], mean_v, rtol=1e-13, atol=1e-13)
            s = w.sm_scale * math.fsum(qf[b, h, R:] * kpe_f)
            assert abs(lse[k] - (s + math.log(L))) < 1e-12


def test_lse_equals_bruteforce_fsum(oracle_mod):
    w = W.make_workload("lse", seed=23, seq_lens=[45, 180], num_heads=3)
    cache = written_cache(oracle_mod, w)
    w.sm_scale = float(np.float32(0.01))  # small |s|, exactly an fp32 value
    _, lse = oracle_decode(oracle_mod, w, cache)
    qf = w.q.to(torch.float64).numpy()
    for b in range(2):
        K = gather_kv(w, cache, b).numpy()
        for h in range(w.num_heads):
            s = [w.sm_scale * math.fsum(qf[b, h] * K[j]) for j in range(K.shape[0])]
            ref = math.log(math.fsum(math.exp(x) for x in s))
            assert abs(lse[b * w.num_heads + h] - ref) < 1e-12


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 8, 64, 300])
def test_split_route_equals_direct(oracle_mod, splits):
    """The split-KV partition (empty splits skipped, including S > L) and its
    LSE merge reach the direct definition up to rounding."""
    w = W.make_workload("split", seed=24, seq_lens=[37, 130, 5, 64], num_heads=4)
    cache = written_cache(oracle_mod, w)
    o0, l0 = oracle_decode(oracle_mod, w, cache)
    o1, l1 = oracle_decode(oracle_mod, w, cache, num_kv_splits=splits)
    np.testing.assert_allclose(o1, o0, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=1e-12, atol=1e-12)


def test_zero_length_sequence(oracle_mod):
    w = W.make_workload("zero", seed=25, seq_lens=[0, 9], num_heads=2, table_pad=1)
    cache = written_cache(oracle_mod, w)
    for splits in (0, 4):
        o, lse = oracle_decode(oracle_mod, w, cache, num_kv_splits=splits)
        assert np.all(o[:2] == 0) and np.all(np.isneginf(lse[:2]))
        assert np.isfinite(o[2:]).all()


def test_out_of_range_block_reads_zeros(oracle_mod):
    w = W.make_workload("oob", seed=26, seq_lens=[100], num_heads=2, pool_blocks=3)
    cache = written_cache(oracle_mod, w)
    spare = [x for x in range(3) if x not in w.block_table[0, :2]][0]
    zero_cache = cache.copy()
    zero_cache[spare] = 0
    bt_good = w.block_table.copy()
    bt_good[0, 1] = spare
    o_ref, l_ref = oracle_mod.decode(w.q, zero_cache, bt_good, w.seq_lens, block_size=64,
                                     kv_lora_rank=512, rope_dim=64, sm_scale=w.sm_scale)
    for bad_id in (-5, 3, 1 << 30):
        bt = w.block_table.copy()
        bt[0, 1] = bad_id
        o, l = oracle_mod.decode(w.q, cache, bt, w.seq_lens, block_size=64, kv_lora_rank=512,
                                 rope_dim=64, sm_scale=w.sm_scale)
        assert np.array_equal(o, o_ref) and np.array_equal(l, l_ref)


def test_pairs_subset_and_thread_count_do_not_change_bits(oracle_mod):
    w = W.make_workload("pairs", seed=27, seq_lens=[100, 60, 20], num_heads=4, rows_per_seq=2)
    cache = written_cache(oracle_mod, w)
    o, lse = oracle_decode(oracle_mod, w, cache, threads=1)
    o4, lse4 = oracle_decode(oracle_mod, w, cache, threads=4)
    assert np.array_equal(o, o4) and np.array_equal(lse, lse4)
    pairs = np.array([[5, 3], [0, 0], [2, 1]])
    op, lp = oracle_decode(oracle_mod, w, cache, pairs=pairs)
    for k, (r, h) in enumerate(pairs):
        assert np.array_equal(op[k], o[r * 4 + h]) and lp[k] == lse[r * 4 + h]


def test_multirow_rows_share_their_sequence(oracle_mod):
    """Rows r*R_ps .. r*R_ps + R_ps - 1 attend to sequence r (no causal mask)."""
    w = W.make_workload("mr", seed=28, seq_lens=[50, 90], num_heads=2, rows_per_seq=3)
    cache = written_cache(oracle_mod, w)
    o, _ = oracle_decode(oracle_mod, w, cache)
    qb = w.q.view(torch.int16).numpy().view(np.uint16)
    for r in range(6):
        single = W.make_workload("mr1", seed=28, seq_lens=[50, 90], num_heads=2)
        single.q = W.bits_to_torch_bf16(np.stack([qb[r], qb[r]]))
        b = r // 3
        o1, _ = oracle_mod.decode(single.q, cache, w.block_table[b:b + 1].repeat(2, 0),
                                  w.seq_lens[b:b + 1].repeat(2), block_size=64,
                                  kv_lora_rank=512, rope_dim=64, sm_scale=w.sm_scale)
        assert np.array_equal(o1[:2], o[r * 2:r * 2 + 2])
