"""GPU parity of MLA decode against the fp64 oracle, plus invariance checks.

Operation: "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
vllm/attention/ops/triton_decode_attention.py (decode_attention_fwd, stage 1
and stage 2) and "Triton and MLA: portable attention and multi-head latent
attention", Data flow (forward_mqa returns o and a natural-log lse).

Bar: |o - ref| <= 1e-2 + 1e-2 |ref| (bf16 output) and |lse - ref| <= 2e-3,
element by element; the cache bytes the decode reads are the ones the GPU
cache write produced, checked byte-exact against the oracle's write.
"""
import numpy as np
import pytest
import torch

import mla_paged_kv_concat_gb300 as mla
from mla_paged_kv_concat_gb300 import workloads as W

from _helpers import (Dev, assert_close, oracle_cache, oracle_decode, sample_pairs,
                      sm_count, unit_pairs)

pytestmark = pytest.mark.gpu

PATHS = [mla.MLA_PATH_MMA_SYNC, mla.MLA_PATH_TCGEN05]


def tc_ok(w):
    """The tcgen05 kernels cover bf16 caches with a 512-wide latent and bf16
    or fp8 caches with a 256-wide latent."""
    return w.kv_lora_rank == 256 or not w.kv_fp8


def _run(w, splits, path=mla.MLA_PATH_AUTO, pairs=None, write=True):
    d = Dev(w)
    if write:
        d.write()
    o, lse = d.decode(splits, path=path)
    torch.cuda.synchronize()
    cache = oracle_cache(w) if write else w.kv_cache
    if write:
        assert d.cache_numpy().tobytes() == cache.tobytes(), "cache write mismatch"
    o_ref, lse_ref = oracle_decode(w, cache, pairs=pairs)
    assert_close(o, lse, o_ref, lse_ref, pairs=pairs, what=f"{w.name} S={splits}")
    return d, o, lse


@pytest.mark.parametrize("splits", [1, 2, 8])
@pytest.mark.parametrize("path", [mla.MLA_PATH_AUTO] + PATHS)
def test_tiny(cuda_dev, splits, path):
    _run(W.make("tiny"), splits, path)


@pytest.mark.parametrize("path", PATHS)
def test_per_shard_forced_kernel(cuda_dev, path):
    """Both stage-1 kernels on the H=16 batch, every (row, head) compared."""
    w = W.make("per_shard")
    _run(w, mla.mla_num_kv_splits(w.max_seq_len, sm_count()), path)


def test_per_shard_full(cuda_dev):
    """B=64, H=16 at the split count the rule gives on this device (the
    benchmark's launch); every (row, head) compared."""
    w = W.make("per_shard")
    S = mla.mla_num_kv_splits(w.max_seq_len, sm_count())
    d, o, lse = _run(w, S)
    assert int(d.err.item()) == 0


@pytest.mark.slow
def test_full_head_sampled(cuda_dev):
    """B=128, H=128 at the benchmark's split count: the first and last query
    vector of every (sequence, 128-vector) unit of the tcgen05 schedule, plus
    random pairs."""
    w = W.make("full_head")
    S = mla.mla_num_kv_splits(w.max_seq_len, sm_count())
    _run(w, S, pairs=unit_pairs(w, 128, extra=32, seed=3))


@pytest.mark.slow
def test_full_head_deterministic_single_pass(cuda_dev):
    w = W.make("full_head")
    d = Dev(w)
    d.write()
    o1, l1 = d.decode(1)
    o1, l1 = o1.clone(), l1.clone()
    o2, l2 = d.decode(1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    pairs = unit_pairs(w, 128, extra=16, seed=4)
    o_ref, lse_ref = oracle_decode(w, oracle_cache(w), pairs=pairs)
    assert_close(o1, l1, o_ref, lse_ref, pairs=pairs, what="full_head S=1")


@pytest.mark.parametrize("path", [mla.MLA_PATH_AUTO] + PATHS)
def test_fp8_small(cuda_dev, path):
    """B=32, H=32, E4M3 cache with R=256 at the benchmark's split count, on
    both stage-1 kernels (AUTO takes the warp-MMA kernel at 32 query
    vectors): the first and last vector of every (sequence, 32-vector) unit
    (each sequence is one 128-vector unit of the tcgen05 schedule), plus
    random pairs."""
    w = W.make("fp8_small")
    S = mla.mla_num_kv_splits(w.max_seq_len, sm_count())
    _run(w, S, path, pairs=unit_pairs(w, 32, extra=64, seed=5))


@pytest.mark.slow
def test_long_multirow_sampled(cuda_dev):
    """8 sequences x 4 rows x 128 heads at the benchmark's split count: the
    first and last vector of each of the 32 (sequence, 128-vector) units of
    the chunked tcgen05 schedule, plus random pairs."""
    w = W.make("long_multirow")
    S = mla.mla_num_kv_splits(w.max_seq_len, sm_count())
    _run(w, S, pairs=unit_pairs(w, 128, extra=8, seed=6))


SMALL = [
    dict(seq_lens=[1, 2, 63, 64, 65, 127, 128, 129], num_heads=16),
    dict(seq_lens=[300, 0, 77], num_heads=16, table_pad=2),
    dict(seq_lens=[200, 130], num_heads=1),
    dict(seq_lens=[200, 130], num_heads=3),
    dict(seq_lens=[190, 70], num_heads=17),
    dict(seq_lens=[333, 64], num_heads=32),
    dict(seq_lens=[150, 257], num_heads=64),
    dict(seq_lens=[150, 257], num_heads=128),
    dict(seq_lens=[260, 100], num_heads=8, rows_per_seq=4),
    dict(seq_lens=[500, 40], num_heads=128, rows_per_seq=2),
    dict(seq_lens=[100, 300], num_heads=16, kv_lora_rank=256),
    dict(seq_lens=[100, 300], num_heads=16, block_size=16),
    dict(seq_lens=[100, 300], num_heads=16, block_size=32),
    dict(seq_lens=[100, 300], num_heads=16, block_size=128),
    dict(seq_lens=[600, 300], num_heads=16, block_size=256),
    dict(seq_lens=[150, 33, 700], num_heads=32, kv_lora_rank=256, kv_fp8=True,
         kv_scale=0.05, write="all"),
    dict(seq_lens=[150, 33], num_heads=16, kv_lora_rank=512, kv_fp8=True,
         kv_scale=0.05, write="all"),
    dict(seq_lens=[90, 1], num_heads=128, kv_lora_rank=256, kv_fp8=True, kv_scale=0.05,
         write="all", block_size=16),
]


@pytest.mark.parametrize("path", [mla.MLA_PATH_AUTO] + PATHS)
@pytest.mark.parametrize("splits", [1, 3, 16])
@pytest.mark.parametrize("case", range(len(SMALL)))
def test_small_shapes(cuda_dev, case, splits, path):
    w = W.make_workload(f"small{case}", seed=200 + case, pool_blocks=None, **SMALL[case])
    if path == mla.MLA_PATH_TCGEN05 and not tc_ok(w):
        pytest.skip("tcgen05 kernels: no fp8 cache with R = 512")
    _run(w, splits, path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("splits", [1, 8])
@pytest.mark.parametrize("q_exp,R,H,rows", [(20, 256, 32, 1), (-30, 512, 16, 1),
                                            (-100, 256, 16, 2), (None, 512, 32, 1),
                                            (None, 256, 128, 1)])
def test_fp8_query_magnitudes(cuda_dev, q_exp, R, H, rows, splits, path):
    """An fp8 cache against queries of extreme magnitude: every element times
    2^q_exp (far outside the fp8 and f16 ranges) with sm_scale times 2^-q_exp
    so that the scores stay moderate, or heads of different magnitudes
    (None: head h times 2^(h mod 5 - 2)).  The query keeps its bf16 range
    through the kernel, so every case matches the oracle."""
    w = W.make_workload(f"fp8q{q_exp}", seed=410 + (q_exp or 0) % 97 + H, pool_blocks=None,
                        seq_lens=[150, 33, 700][: 3 - rows + 1], num_heads=H,
                        rows_per_seq=rows, kv_lora_rank=R, kv_fp8=True, kv_scale=0.05,
                        write="all")
    q = w.q.double()
    if q_exp is None:
        q = q * (2.0 ** (torch.arange(H, dtype=torch.float64) % 5 - 2))[None, :, None]
        sm = w.sm_scale
    else:
        q = q * 2.0 ** q_exp
        sm = float(np.float32(w.sm_scale) * np.float32(2.0 ** -q_exp))
    q32 = q.float()
    assert torch.isfinite(q32).all()
    w.q = q32.bfloat16()
    assert torch.equal(w.q.double(), q)  # power-of-two scaling is exact in bf16
    w.sm_scale = sm
    if path == mla.MLA_PATH_TCGEN05 and not tc_ok(w):
        pytest.skip("tcgen05 kernels: no fp8 cache with R = 512")
    _run(w, splits, path)


@pytest.mark.parametrize("path", PATHS)
def test_forced_kernel_rejects_what_it_does_not_cover(cuda_dev, path):
    """An fp8 cache with a 512-wide latent has no tcgen05 kernel: forcing one
    is refused before any launch; the warp-MMA kernel covers it."""
    w = W.make_workload("rej", seed=64, seq_lens=[100], num_heads=16, kv_fp8=True,
                        kv_scale=0.05, write="all")
    d = Dev(w)
    d.write()
    if path == mla.MLA_PATH_TCGEN05:
        with pytest.raises(mla.MlaError):
            d.decode(2, path=path)
    else:
        d.decode(2, path=path)


def test_padded_block_stride(cuda_dev):
    """A cache whose blocks are further apart than block_size * D."""
    w = W.make_workload("stride", seed=60, seq_lens=[190, 64], num_heads=16, pool_blocks=6)
    d = Dev(w)
    d.write()
    nb, bs, D = w.kv_cache.shape
    big = torch.full((nb, bs * D + 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    big[:, :bs * D] = d.cache.reshape(nb, bs * D)
    view = big[:, :bs * D].view(nb, bs, D)
    o, lse = mla.decode(d.q, view, d.block_table, d.seq_lens, w.sm_scale, 2)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_decode(w, oracle_cache(w))
    assert_close(o, lse, o_ref, lse_ref, what="padded stride")


@pytest.mark.parametrize("H,path", [(16, mla.MLA_PATH_MMA_SYNC), (32, mla.MLA_PATH_MMA_SYNC),
                                    (8, mla.MLA_PATH_MMA_SYNC), (128, mla.MLA_PATH_TCGEN05)])
def test_strided_q(cuda_dev, H, path):
    """q as a view with padded heads and padded rows (head stride 640, row
    stride (H + 2) * 640 elements): the tensor-map and the gathered Q loads
    must both follow the strides."""
    w = W.make_workload("qstride", seed=65, seq_lens=[190, 64, 301], num_heads=H)
    d = Dev(w)
    d.write()
    rows, D = w.num_rows, w.head_dim
    big = torch.full((rows, H + 2, 640), float("nan"), dtype=torch.bfloat16, device="cuda")
    big[:, :H, :D] = d.q
    q_view = big[:, :H, :D]
    assert q_view.stride(1) == 640 and q_view.stride(0) == (H + 2) * 640
    for splits in (1, 3):
        o, lse = mla.decode(q_view, d.cache, d.block_table, d.seq_lens, w.sm_scale, splits,
                            path=path)
        torch.cuda.synchronize()
        o_ref, lse_ref = oracle_decode(w, oracle_cache(w))
        assert_close(o, lse, o_ref, lse_ref, what=f"strided q H={H} S={splits}")


def test_split_count_does_not_change_result_beyond_rounding(cuda_dev):
    w = W.make("per_shard")
    d = Dev(w)
    d.write()
    o1, l1 = d.decode(1)
    o1 = o1.float()
    for S in (2, 5, 8, 64):
        o, l = d.decode(S)
        assert torch.allclose(o.float(), o1, atol=1e-2, rtol=1e-2)
        assert torch.allclose(l, l1, atol=2e-3)


@pytest.mark.parametrize("path", PATHS)
def test_repeat_runs_bitwise_equal(cuda_dev, path):
    w = W.make("per_shard")
    d = Dev(w)
    d.write()
    for S in (1, 8):
        a = [t.clone() for t in d.decode(S, path=path)]
        b = d.decode(S, path=path)
        torch.cuda.synchronize()
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("path", PATHS)
def test_single_pass_is_batch_invariant(cuda_dev, path):
    """With one split, a row's result does not depend on the rest of the batch."""
    w = W.make("per_shard")
    d = Dev(w)
    d.write()
    o_all, l_all = d.decode(1, path=path)
    for b in (0, 17, 63):
        o_b, l_b = mla.decode(d.q[b:b + 1], d.cache, d.block_table[b:b + 1],
                              d.seq_lens[b:b + 1], w.sm_scale, 1, path=path)
        torch.cuda.synchronize()
        assert torch.equal(o_b[0], o_all[b]) and torch.equal(l_b[0], l_all[b])


@pytest.mark.parametrize("path,R,fp8", [(mla.MLA_PATH_MMA_SYNC, 512, False),
                                         (mla.MLA_PATH_TCGEN05, 512, False),
                                         (mla.MLA_PATH_TCGEN05, 256, True)])
def test_physical_block_permutation_is_bitwise_invariant(cuda_dev, path, R, fp8):
    """Moving every block to another physical slot (and rewriting the table)
    leaves the output bit-for-bit unchanged (the paged-layout invariance of
    the pages' test_decode_attention, page size 1 vs 16)."""
    kw = dict(kv_fp8=True, kv_scale=0.05, write="all") if fp8 else {}
    w = W.make_workload("perm", seed=61, seq_lens=[700, 129, 64], num_heads=16,
                        pool_blocks=30, kv_lora_rank=R, **kw)
    d = Dev(w)
    d.write()
    o1, l1 = [t.clone() for t in d.decode(4, path=path)]
    perm = torch.randperm(30, generator=torch.Generator().manual_seed(0)).cuda()
    new_cache = torch.empty_like(d.cache)
    new_cache[perm] = d.cache
    new_bt = perm[d.block_table.long()].int()
    o2, l2 = mla.decode(d.q, new_cache, new_bt, d.seq_lens, w.sm_scale, 4, path=path,
                        kv_lora_rank=R, kv_scale=d.kv_scale if fp8 else None)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_out_of_range_block_id_reads_zeros_and_counts(cuda_dev):
    w = W.make_workload("oob", seed=62, seq_lens=[100, 70], num_heads=16, pool_blocks=5)
    d = Dev(w)
    d.write()
    bt = w.block_table.copy()
    bt[0, 1] = 1 << 20
    bt[1, 1] = -3
    w.block_table = bt
    d.block_table = torch.from_numpy(bt).cuda()
    d.err.zero_()
    o, lse = d.decode(2)
    torch.cuda.synchronize()
    assert int(d.err.item()) >= 2
    o_ref, lse_ref = oracle_decode(w, oracle_cache(w))
    assert_close(o, lse, o_ref, lse_ref, what="oob")


def test_seq_len_beyond_table_is_clamped_and_counted(cuda_dev):
    w = W.make_workload("clamp", seed=63, seq_lens=[128], num_heads=16, pool_blocks=3)
    d = Dev(w)
    d.write()
    d.seq_lens = torch.tensor([1000], dtype=torch.int32, device="cuda")
    d.err.zero_()
    o, lse = d.decode(1)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 1
    o_ref, lse_ref = oracle_decode(w, oracle_cache(w))
    assert_close(o, lse, o_ref, lse_ref, what="clamp")


@pytest.mark.parametrize("path", PATHS)
def test_split_count_at_its_cap(cuda_dev, path):
    """The split rule's cap, 2 x SMs, reached by a 160k-token sequence next to
    short ones (most of the 304 slots of the short rows stay unused); every
    (row, head) compared."""
    H = 16 if path == mla.MLA_PATH_MMA_SYNC else 128
    w = W.make_workload("cap", seed=77, seq_lens=[160_000, 3, 700], num_heads=H,
                        pool_blocks=2600)
    S = mla.mla_num_kv_splits(w.max_seq_len, sm_count())
    assert S == 2 * sm_count()
    pairs = None if H == 16 else unit_pairs(w, 128, extra=32, seed=8)
    d, o, lse = _run(w, S, path, pairs=pairs)
    assert int(d.err.item()) == 0


@pytest.mark.parametrize("path", PATHS)
def test_many_splits_on_short_sequences(cuda_dev, path):
    """More split slots than tiles: every row's unused slots are marked and
    skipped by the merge."""
    H = 16 if path == mla.MLA_PATH_MMA_SYNC else 128
    w = W.make_workload("shortS", seed=78, seq_lens=[1, 64, 65, 200, 0], num_heads=H)
    _run(w, 2 * sm_count(), path)


@pytest.mark.parametrize("R,fp8", [(512, False), (256, False), (256, True), (512, True)])
@pytest.mark.parametrize("H,rows", [(32, 1), (33, 1), (16, 2), (17, 2)])
def test_auto_kernel_choice(cuda_dev, R, fp8, H, rows):
    """AUTO runs the tcgen05 kernel above 32 query vectors per sequence when
    one covers the cache (R = 512 bf16, R = 256 bf16 or fp8) and the
    warp-MMA kernel otherwise: its result is bitwise that of the forced
    choice, and it meets the decode bar against the oracle."""
    w = W.make_workload("auto", seed=41 + H + R, seq_lens=[700, 130, 1], num_heads=H,
                        kv_lora_rank=R, rows_per_seq=rows,
                        **(dict(kv_fp8=True, kv_scale=0.05, write="all") if fp8 else {}))
    S = 4
    d = Dev(w)
    d.write()
    o_auto, l_auto = d.decode(S, path=mla.MLA_PATH_AUTO)
    tc = H * rows > 32 and (R == 256 or not fp8)
    o_ref_path, l_ref_path = d.decode(S, path=mla.MLA_PATH_TCGEN05 if tc else mla.MLA_PATH_MMA_SYNC)
    torch.cuda.synchronize()
    assert torch.equal(o_auto.view(torch.int16), o_ref_path.view(torch.int16))
    assert torch.equal(l_auto, l_ref_path)
    o_ref, lse_ref = oracle_decode(w, oracle_cache(w))
    assert_close(o_auto, l_auto, o_ref, lse_ref, what=f"AUTO H={H} rows={rows} R={R} fp8={fp8}")


@pytest.mark.parametrize("H,R,fp8,path", [
    (128, 512, False, mla.MLA_PATH_TCGEN05),
    (128, 256, True, mla.MLA_PATH_TCGEN05),
    (16, 512, False, mla.MLA_PATH_MMA_SYNC),
])
def test_more_units_than_the_persistent_schedule_holds(cuda_dev, H, R, fp8, path):
    """520 sequences of one vector block each: more (sequence, block) units
    than the persistent schedules hold (512), so stage 1 runs as a grid of
    (block, split group) CTAs (pairs) with S = 4.  Lengths 1..300, some of
    them shorter than a split.  The first and last vector of every unit and
    random pairs against the oracle."""
    from _helpers import unit_pairs
    rng = np.random.default_rng(77)
    lens = rng.integers(1, 301, size=520)
    kw = dict(kv_fp8=True, kv_scale=0.05, write="all") if fp8 else {}
    w = W.make_workload("grid", seed=78 + H + R, seq_lens=lens, num_heads=H, kv_lora_rank=R,
                        **kw)
    pairs = unit_pairs(w, 128 if H == 128 else 16, extra=64, seed=3)
    _run(w, 4, path, pairs=pairs)
