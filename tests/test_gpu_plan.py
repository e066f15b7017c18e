"""GPU parity of the query given as the (q_nope, q_pe) pair and of decode
plans, including a plan captured into a CUDA graph and replayed over new
buffer contents.

Operation: "Triton and MLA: portable attention and multi-head latent
attention", Data flow (forward_mqa takes q as a tensor or a (q_nope, q_pe)
tuple) and "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
vllm/attention/backends/triton_mla.py, TritonMLAState (decode captured once
over fixed slot_mapping / seq_lens / block_tables buffers, replayed after
their contents are refreshed).

Bar: the pair gives the same bits as the concatenated q (same kernels, same
schedule); plans and replays meet the decode bar against the oracle
(|o - ref| <= 1e-2 + 1e-2 |ref|, |lse - ref| <= 2e-3) and write the cache
byte-exact (plain write) or as the fused write's test allows.
"""
import numpy as np
import pytest
import torch

import mla_paged_kv_concat_gb300 as mla
import oracle
from mla_paged_kv_concat_gb300 import workloads as W

from _helpers import Dev, assert_close, oracle_cache, oracle_decode, sm_count

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("H,R,path", [
    (16, 512, mla.MLA_PATH_MMA_SYNC), (3, 512, mla.MLA_PATH_MMA_SYNC),
    (32, 256, mla.MLA_PATH_MMA_SYNC), (128, 512, mla.MLA_PATH_TCGEN05),
    (128, 512, mla.MLA_PATH_MMA_SYNC),
])
@pytest.mark.parametrize("splits", [1, 4])
def test_q_pair_equals_concatenated_q(cuda_dev, H, R, path, splits):
    w = W.make_workload("qpair", seed=91 + H, seq_lens=[300, 1000, 77, 1], num_heads=H,
                        kv_lora_rank=R)
    d = Dev(w)
    d.write()
    o1, l1 = d.decode(splits, path=path)
    q_nope = d.q[:, :, :R].clone()
    # q_pe with a padded head stride (96 elements)
    q_pe = torch.zeros(w.num_rows, H, 96, dtype=torch.bfloat16, device="cuda")[:, :, :64]
    q_pe.copy_(d.q[:, :, R:])
    o2, l2 = mla.decode((q_nope, q_pe), d.cache, d.block_table, d.seq_lens, w.sm_scale, splits,
                        err_count=d.err, path=path)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
    o_ref, lse_ref = oracle_decode(w, oracle_cache(w))
    assert_close(o2, l2, o_ref, lse_ref, what=f"q pair H={H}")


def _device(w):
    d = Dev(w)
    return d


def _norm_rope_dev(x):
    return dict(gamma=x.gamma.cuda(), eps=x.eps, positions=torch.from_numpy(x.positions).cuda(),
                cos_sin_table=torch.from_numpy(x.table).cuda())


def _reference(w, x=None, rotate_q=False):
    """Oracle cache after the step's write, and the oracle decode after it."""
    cache = w.kv_cache.copy()
    q_bits = _bits(w.q).copy()
    if x is None:
        oracle.cache_write(w.kv_c, w.k_pe, w.slot_mapping, cache, block_size=w.block_size,
                           kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim, kv_is_fp8=False)
    else:
        oracle.norm_rope_cache_write(
            w.kv_c, w.k_pe, x.gamma, x.eps, x.positions, x.table, w.slot_mapping, cache,
            block_size=w.block_size, kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim,
            kv_is_fp8=False, q_pe=q_bits[:, :, w.kv_lora_rank:] if rotate_q else None)
    w2 = W.Workload(**{**w.__dict__, "q": W.bits_to_torch_bf16(q_bits)})
    return cache, oracle_decode(w2, cache)


@pytest.mark.parametrize("H", [16, 128])
@pytest.mark.parametrize("fused", [False, True])
def test_plan_runs_the_step(cuda_dev, H, fused):
    w = W.make_workload("plan", seed=95 + H, seq_lens=[300, 1000, 77, 640], num_heads=H)
    x = W.norm_rope_inputs(w, seed=9) if fused else None
    d = _device(w)
    plan = mla.DecodePlan(d.q, d.cache, d.block_table, d.seq_lens, w.sm_scale,
                          mla.mla_num_kv_splits(w.max_seq_len, sm_count()), err_count=d.err,
                          write=dict(kv_c=d.kv_c, k_pe=d.k_pe, slot_mapping=d.slot_mapping),
                          norm_rope=dict(_norm_rope_dev(x), rotate_q=True) if fused else None)
    o, lse = plan.run()
    torch.cuda.synchronize()
    plan.close()
    assert int(d.err.item()) == 0
    cache_ref, (o_ref, lse_ref) = _reference(w, x, rotate_q=fused)
    if not fused:
        assert d.cache_numpy().tobytes() == cache_ref.tobytes()
    assert_close(o, lse, o_ref, lse_ref, what=f"plan H={H} fused={fused}")


@pytest.mark.parametrize("H,fused,pair", [(16, False, False), (128, False, True),
                                          (16, True, True), (128, True, False)])
def test_plan_graph_replay_over_new_contents(cuda_dev, H, fused, pair):
    """Capture plan.run() once, then refresh every buffer's contents (new
    lengths, block ids, queries, new tokens, positions) and replay."""
    bs, maxb, pool = 64, 24, 120
    cap = maxb * bs

    def make(seed, lens):
        w = W.make_workload("graph", seed=seed, seq_lens=lens, num_heads=H, pool_blocks=pool,
                            table_pad=maxb - max((int(L) + bs - 1) // bs for L in lens))
        assert w.block_table.shape == (len(lens), maxb)
        return w

    w1 = make(101, [300, 1000, 77, 640, 1500])
    w2 = make(102, [1200, 5, 900, 64, cap])
    S = mla.mla_num_kv_splits(cap, sm_count())
    xs = [W.norm_rope_inputs(w, seed=12, max_position=cap + 64) if fused else None
          for w in (w1, w2)]
    d = _device(w1)
    R = w1.kv_lora_rank
    if pair:
        q_nope = d.q[:, :, :R].clone()
        q_pe = d.q[:, :, R:].clone()
    nr = _norm_rope_dev(xs[0]) if fused else None
    plan = mla.DecodePlan(q_nope if pair else d.q, d.cache, d.block_table, d.seq_lens,
                          w1.sm_scale, S, q_pe=q_pe if pair else None, err_count=d.err,
                          write=dict(kv_c=d.kv_c, k_pe=d.k_pe, slot_mapping=d.slot_mapping),
                          norm_rope=dict(nr, rotate_q=True) if fused else None)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        plan.run()          # first run outside the capture (kernel attributes)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.run()

    def load(w, x):
        d.cache.copy_(Dev(w).cache)
        if pair:
            q_nope.copy_(w.q[:, :, :R])
            q_pe.copy_(w.q[:, :, R:])
        else:
            d.q.copy_(w.q)
        d.block_table.copy_(torch.from_numpy(w.block_table))
        d.seq_lens.copy_(torch.from_numpy(w.seq_lens))
        d.kv_c.copy_(w.kv_c)
        d.k_pe.copy_(w.k_pe)
        d.slot_mapping.copy_(torch.from_numpy(w.slot_mapping))
        if x is not None:
            nr["gamma"].copy_(x.gamma)
            nr["positions"].copy_(torch.from_numpy(x.positions))
            nr["cos_sin_table"].copy_(torch.from_numpy(x.table))
        d.err.zero_()

    for w, x in ((w2, xs[1]), (w1, xs[0])):
        load(w, x)
        g.replay()
        torch.cuda.synchronize()
        assert int(d.err.item()) == 0
        cache_ref, (o_ref, lse_ref) = _reference(w, x, rotate_q=fused)
        if not fused:
            assert d.cache_numpy().tobytes() == cache_ref.tobytes()
        assert_close(plan.out, plan.lse, o_ref, lse_ref, what=f"replay H={H} L={w.seq_lens}")
    plan.close()


@pytest.mark.parametrize("name,unit", [("per_shard", 16), ("full_head", 128),
                                       ("long_multirow", 128)])
def test_benchmark_configuration_through_a_plan(cuda_dev, name, unit):
    """The benchmark's step as it times it: one plan over the resident
    tensors (write of the new tokens, stage 1 at the rule's split count,
    merge), run once; the cache compared byte for byte and, against the
    oracle, the first and last (row, head) of every stage-1 unit (`unit`
    query vectors of one sequence) plus random pairs."""
    from _helpers import unit_pairs
    w = W.make(name)
    d = _device(w)
    S = mla.mla_num_kv_splits(w.max_seq_len, sm_count())
    plan = mla.DecodePlan(d.q, d.cache, d.block_table, d.seq_lens, w.sm_scale, S,
                          err_count=d.err,
                          write=dict(kv_c=d.kv_c, k_pe=d.k_pe, slot_mapping=d.slot_mapping))
    o, lse = plan.run()
    torch.cuda.synchronize()
    plan.close()
    assert int(d.err.item()) == 0
    cache = oracle_cache(w)
    assert d.cache_numpy().tobytes() == cache.tobytes()
    pairs = unit_pairs(w, unit, extra=32, seed=11)
    o_ref, lse_ref = oracle_decode(w, cache, pairs=pairs)
    assert_close(o, lse, o_ref, lse_ref, pairs=pairs, what=f"{name} through a plan")
