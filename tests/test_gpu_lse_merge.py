"""GPU parity of the cross-shard LSE merge (decode context parallelism).

Operation: "Triton and MLA: portable attention and multi-head latent
attention", Design motivation (decode returns lse so that the per-shard
(o, lse) pairs of decode context parallelism can be merged,
cp_lse_ag_out_rs), with the LSE algebra of "frozenleaves/vllm compare
v0.11.0...mla_cuda_graphs", vllm/attention/ops/triton_decode_attention.py,
_fwd_kernel_stage2.

Two checks: (1) random bf16 parts with random lse (empty parts, records with
no tokens at all, more than 32 parts) against the oracle's merge of the same
bf16 values, element by element; the only rounding beyond fp32 is the bf16
output, so |o - ref| <= 1e-3 + 4e-3 |ref| and |lse - ref| <= 1e-4.
(2) A sharded decode: each sequence's tokens cut into G contiguous page
ranges, each shard decoded on the GPU, the shards merged on the GPU, compared
with the oracle's direct decode of the whole sequences at the decode bar
(|o - ref| <= 1e-2 + 1e-2 |ref|, |lse - ref| <= 2e-3).
"""
import numpy as np
import pytest
import torch

import mla_paged_kv_concat_gb300 as mla
import oracle
from mla_paged_kv_concat_gb300 import workloads as W

from _helpers import Dev, assert_close, oracle_cache, oracle_decode, sm_count

pytestmark = pytest.mark.gpu


def _random_parts(G, rows, H, R, seed):
    rng = np.random.default_rng(seed)
    n = rows * H
    o = torch.from_numpy(rng.standard_normal((G, rows, H, R)).astype(np.float32)).to(
        torch.bfloat16)
    lse = (rng.standard_normal((G, n)) * 4.0 + 2.0).astype(np.float32)
    lse[rng.random((G, n)) < 0.3] = -np.inf
    lse[:, 0] = -np.inf                      # a record with no tokens in any part
    if n > 1:
        lse[:, 1] = -np.inf
        lse[G - 1, 1] = 0.75                 # a record held by one part only
    if n > 2:
        lse[:, 2] = np.linspace(-60.0, 60.0, G)  # weights spanning e^120
    return o, lse.reshape(G, rows, H)


@pytest.mark.parametrize("G,rows,H,R", [
    (1, 3, 16, 512), (2, 5, 16, 512), (3, 4, 128, 512), (7, 2, 16, 256),
    (32, 2, 8, 512), (40, 2, 8, 512), (33, 1, 128, 256), (4, 64, 16, 512),
])
def test_random_parts_match_oracle(cuda_dev, G, rows, H, R):
    o_parts, lse_parts = _random_parts(G, rows, H, R, seed=G * 1000 + rows * 10 + H + R)
    o_d, lse_d = mla.lse_merge(o_parts.cuda(), torch.from_numpy(lse_parts).cuda())
    torch.cuda.synchronize()
    n = rows * H
    o_ref, lse_ref = oracle.lse_merge(
        o_parts.float().numpy().astype(np.float64).reshape(G, n, R),
        lse_parts.astype(np.float64).reshape(G, n))
    og = o_d.float().cpu().numpy().astype(np.float64).reshape(n, R)
    lg = lse_d.cpu().numpy().astype(np.float64).reshape(n)
    err = np.abs(og - o_ref)
    bad = ~(err <= 1e-3 + 4e-3 * np.abs(o_ref))
    assert not bad.any(), (np.argwhere(bad)[:5].tolist(), float(np.nanmax(err)))
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), empty)
    assert np.all(og[empty] == 0.0)
    assert np.all(np.abs(lg[~empty] - lse_ref[~empty]) <= 1e-4)


def test_zero_rows_is_a_noop(cuda_dev):
    o, lse = mla.lse_merge(torch.empty(3, 0, 16, 512, dtype=torch.bfloat16, device="cuda"),
                           torch.empty(3, 0, 16, dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert o.shape == (0, 16, 512) and lse.shape == (0, 16)


def _shard_tables(w, cuts):
    """Per shard: (block_table, seq_lens) covering the token range
    [cuts[b, g], cuts[b, g+1]) of every sequence b (cuts on page boundaries)."""
    bs = w.block_size
    B = w.num_seqs
    out = []
    for g in range(cuts.shape[1] - 1):
        bt = np.zeros_like(w.block_table)
        sl = np.zeros(B, np.int32)
        for b in range(B):
            a, z = int(cuts[b, g]), int(cuts[b, g + 1])
            m = (z - a + bs - 1) // bs
            bt[b, :m] = w.block_table[b, a // bs:a // bs + m]
            bt[b, m:] = w.block_table[b, -1]
            sl[b] = z - a
        out.append((bt, sl))
    return out


@pytest.mark.parametrize("G,H,seed", [(2, 16, 1), (3, 128, 2), (4, 16, 3), (5, 64, 4)])
def test_sharded_decode_then_merge(cuda_dev, G, H, seed):
    w = W.make_workload("dcp", seed=90 + seed, seq_lens=[130, 257, 64, 700, 1500, 1],
                        num_heads=H)
    d = Dev(w)
    d.write()
    rng = np.random.default_rng(seed)
    bs = w.block_size
    cuts = np.zeros((w.num_seqs, G + 1), np.int64)
    for b, L in enumerate(w.seq_lens):
        pages = (int(L) + bs - 1) // bs
        inner = np.sort(rng.integers(0, pages + 1, size=G - 1)) * bs  # empty shards allowed
        cuts[b] = np.concatenate([[0], np.minimum(inner, L), [L]])
    o_parts = torch.empty(G, w.num_rows, H, w.kv_lora_rank, dtype=torch.bfloat16,
                          device="cuda")
    lse_parts = torch.empty(G, w.num_rows, H, dtype=torch.float32, device="cuda")
    for g, (bt, sl) in enumerate(_shard_tables(w, cuts)):
        S = mla.mla_num_kv_splits(int(sl.max()), sm_count())
        mla.decode(d.q, d.cache, torch.from_numpy(bt).cuda(), torch.from_numpy(sl).cuda(),
                   w.sm_scale, S, kv_lora_rank=w.kv_lora_rank, err_count=d.err,
                   out=o_parts[g], lse=lse_parts[g])
    o, lse = mla.lse_merge(o_parts, lse_parts)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    o_ref, lse_ref = oracle_decode(w, oracle_cache(w))
    assert_close(o, lse, o_ref, lse_ref, what=f"dcp G={G} H={H}")
