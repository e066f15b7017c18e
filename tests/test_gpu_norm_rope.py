"""GPU parity of the fused RMSNorm + rotary + cache write against the oracle.

Operation: "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
vllm/model_executor/models/deepseek_v2.py (kv_a_layernorm = RMSNorm;
rotary_emb = get_rope(..., is_neox_style=False)) and the MLA common forward
(q_pe and k_pe rotated by position, then concat_and_cache_mla).

Bar: bit-exact.  The oracle evaluates the RMSNorm and the rotation in fp64
and rounds once to bf16; the kernel reaches the same bits (double-float
evaluation with an error band, the fp64 operation sequence next to a
rounding midpoint), so the cache bytes (bf16 and fp8) and the rotated q_pe
must equal the oracle's.  Crafted rows put exact ties and near-ties on the
fp64 path and on the band's edge; edge values (NaN, infinities, zeros,
subnormals, huge values, eps = 0) are covered too.  Everything not written
(padded slots, skipped tokens, the rest of the pool) is compared byte for
byte, and skipped tokens are counted exactly.
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


def _check_bf16(got_bits, ref_bits, what=""):
    bad = np.asarray(got_bits) != np.asarray(ref_bits)
    assert not bad.any(), (what, int(bad.sum()), np.argwhere(bad)[:5].tolist(),
                           np.asarray(got_bits)[bad][:5], np.asarray(ref_bits)[bad][:5])


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
    """The whole cache, byte for byte (written rows, skipped tokens, the rest
    of the pool)."""
    D = w.head_dim
    got = d.cache_numpy().reshape(-1, D)
    ref = cache_ref.reshape(-1, D)
    bad = np.any(got != ref, axis=1)
    assert not bad.any(), (f"{int(bad.sum())} cache rows differ", np.argwhere(bad)[:5].tolist())


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
    _check_bf16(_bits(q_pe), q_ref, what="rotated q_pe")
    bad = (x.positions < 0) | (x.positions >= x.table.shape[0])
    assert np.array_equal(_bits(q_pe)[bad], q_in[bad])


def test_scaled_table_and_q_pe_as_rope_columns_of_q(cuda_dev):
    """A table with a magnitude factor (as the YaRN scale would give) and q_pe
    given as the rope columns of q (head stride R+P, row stride H(R+P))."""
    w = W.make_workload("nr_view", seed=82, seq_lens=[300, 1000, 77, 64], num_heads=16)
    x = W.norm_rope_inputs(w, seed=6, table_scale=1.25)
    d, cache_ref, q_pe, q_ref = _run(w, x, fp8=False, q_pe_view=True)
    _compare_cache(w, x, d, cache_ref, False)
    _check_bf16(_bits(q_pe), q_ref, what="q rope cols")


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


def _bf16(vals) -> np.ndarray:
    """bf16 bits of values that bf16 holds exactly."""
    v = np.asarray(vals, np.float32)
    b = W.bf16_bits_from_f32(v)
    back = W.bits_to_torch_bf16(b).float().numpy()
    assert np.array_equal(back.view(np.uint32), v.view(np.uint32)) | np.isnan(v).all(), vals
    return b


def _crafted(R: int, H: int, seed: int):
    """Rows whose RMSNorm or rotation lands exactly on a bf16 rounding midpoint
    (the fp64 path must take over and round to even), next to one (the band
    test must decide from the low part), and edge values.

    RMSNorm ties: a row of +-1 with one element +-35 has sum of squares
    S = 1225 + (R - 1); with eps = (25 R - S) / R (exact in fp32) the mean
    square plus eps is exactly 25, so 1 / sqrt(.) = 0.2 and the reference
    gives fl(35 * fl(0.2)) = 7 exactly, then 7 * gamma; gamma = 37/256,
    73/512 and 55/256 give 259/256, 511/512 and 385/256, each halfway between
    two bf16 values.  Rotation ties: cos = 1 + 2^-8, sin = 0 on the pair
    (1, 1); near-ties 2^-30 either side of a midpoint: cos = 1 + 2^-8,
    sin = 2^-20 on (1, +-2^-10)."""
    rng = np.random.default_rng(seed)
    S = 1225 + (R - 1)
    eps = float(np.float32((25 * R - S) / R))
    assert eps == (25 * R - S) / R
    tie_d = [3, 100, 201, R - 2]
    tie_g = [37 / 256, 73 / 512, 55 / 256, -37 / 256]
    gamma = (1.0 + 0.25 * rng.standard_normal(R)).astype(np.float32)
    gamma = W.bits_to_torch_bf16(W.bf16_bits_from_f32(gamma)).float().numpy()
    for d, g in zip(tie_d, tie_g):
        gamma[d] = g
    gamma[[7, 8, 9, 10]] = [0.0, -0.0, 2.0 ** -120, 2.0 ** 100]
    rows = []
    # ties: +-35 at a tie element, +-1 elsewhere
    for i, d in enumerate(tie_d * 2):
        r = rng.choice([-1.0, 1.0], size=R).astype(np.float32)
        r[d] = 35.0 if i < len(tie_d) else -35.0
        rows.append(r)
    # random rows (fast path with this eps)
    for _ in range(6):
        rows.append(rng.standard_normal(R).astype(np.float32))
    # edge rows
    z = np.zeros(R, np.float32)
    r = rng.standard_normal(R).astype(np.float32); r[5] = np.nan; rows.append(r)
    r = rng.standard_normal(R).astype(np.float32); r[6] = np.inf; rows.append(r)
    rows.append(z.copy())                                   # all zero
    r = z.copy(); r[::3] = -0.0; rows.append(r)             # signed zeros
    rows.append((rng.integers(1, 127, size=R) * 2.0 ** -133).astype(np.float32))  # subnormals
    rows.append((rng.choice([-1.0, 1.0], size=R) * 2.0 ** 126 *
                 (1 + rng.integers(0, 127, size=R) / 128)).astype(np.float32))    # huge
    r = (rng.standard_normal(R) * 2.0 ** -60).astype(np.float32); r[11] = 2.0 ** 40
    rows.append(r)                                          # wide range
    r = rng.standard_normal(R).astype(np.float32) * 1e-3; r[0] = 2.0 ** -20; rows.append(r)
    kv_c = np.stack([W.bits_to_torch_bf16(W.bf16_bits_from_f32(x)).float().numpy()
                     for x in rows])
    T = kv_c.shape[0]
    # rotation table rows: crafted positions 0..5, random after
    P = 64
    npos = 16
    ang = rng.uniform(0, 2 * np.pi, size=(npos, P // 2))
    table = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    h = P // 2
    table[0, :h], table[0, h:] = 1 + 2.0 ** -8, 0.0        # exact ties on (1, 1)
    table[1, :h], table[1, h:] = 1 + 2.0 ** -8, 2.0 ** -20  # near-ties on (1, +-2^-10)
    table[2, :h], table[2, h:] = 1.0, 1.0                   # (a, -a): exact zero
    table[3, 0] = np.nan                                    # NaN angle for pair 0
    table[4, :h], table[4, h:] = 2.0 ** -110, 2.0 ** -110   # tiny products
    table[5, :h], table[5, h:] = 2.0 ** 100, -(2.0 ** 100)  # huge products
    pos = rng.integers(0, npos, size=T).astype(np.int64)
    pos[:6] = np.arange(6)

    def pe_rows(n):
        x = rng.standard_normal((n, P)).astype(np.float32)
        x = W.bits_to_torch_bf16(W.bf16_bits_from_f32(x)).float().numpy()
        for t in range(n):
            p = pos[t] if n == T else None
            if p == 0:
                x[t] = 1.0
            elif p == 1:
                x[t, 0::2] = 1.0
                x[t, 1::2] = np.where(np.arange(h) % 2 == 0, 2.0 ** -10, -(2.0 ** -10))
            elif p == 2:
                x[t, 1::2] = -x[t, 0::2]
        return x
    k_pe = pe_rows(T)
    q_pe = np.stack([pe_rows(T) for _ in range(H)], axis=1)  # [T, H, P]
    q_pe[:, H // 2:] = W.bits_to_torch_bf16(W.bf16_bits_from_f32(
        rng.standard_normal((T, H - H // 2, P)).astype(np.float32))).float().numpy()
    return dict(kv_c=kv_c, k_pe=k_pe, gamma=gamma, eps=eps, table=table, positions=pos,
                q_pe=q_pe)


def _nan_code(c, fmt):
    c = c.astype(np.int32) & 0x7F
    return c == 0x7F if fmt == "e4m3" else c > 0x7C


@pytest.mark.parametrize("R,fmt", [(512, None), (256, None), (512, "e4m3"), (256, "e5m2")])
def test_fused_write_exact_ties_and_edges(cuda_dev, R, fmt):
    """Crafted exact ties, near-ties and edge values through the fused write:
    cache (bf16, or fp8 of the rounded bf16 values) and rotated q_pe equal the
    oracle bit for bit (for fp8, a NaN code wherever the oracle has one)."""
    H = 4
    c = _crafted(R, H, seed=R + (0 if fmt is None else 7))
    T = c["kv_c"].shape[0]
    fp8 = fmt is not None
    w = W.make_workload(f"ties{R}", seed=95, seq_lens=[T], num_heads=H, kv_lora_rank=R,
                        pool_blocks=4, write="random", num_write_tokens=T, poison=False)
    w.slot_mapping = np.arange(T, dtype=np.int64) + 3
    w.kv_c = W.bits_to_torch_bf16(_bf16(c["kv_c"]))
    w.k_pe = W.bits_to_torch_bf16(_bf16(c["k_pe"]))
    if fp8:
        w.kv_fp8, w.kv_scale = True, float(np.float32(0.25))
        w.kv_cache = np.zeros(w.kv_cache.shape, np.uint8)
    gamma = W.bits_to_torch_bf16(_bf16(c["gamma"]))
    q_pe_t = W.bits_to_torch_bf16(_bf16(c["q_pe"]))
    d = Dev(w)
    q_pe = q_pe_t.cuda()
    kv_dtype = {None: None, "e4m3": "fp8_e4m3", "e5m2": "fp8_e5m2"}[fmt]
    mla.norm_rope_cache_write(d.kv_c, d.k_pe, d.cache, d.slot_mapping, gamma.cuda(), c["eps"],
                              torch.from_numpy(c["positions"]).cuda(),
                              torch.from_numpy(c["table"]).cuda(), q_pe=q_pe,
                              kv_cache_dtype=kv_dtype, scale=d.kv_scale if fp8 else None,
                              err_count=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    cache_ref = w.kv_cache.copy()
    q_ref = _bits(q_pe_t).copy()
    kw = dict(fp8_format=fmt) if fp8 else {}
    oracle.norm_rope_cache_write(w.kv_c, w.k_pe, gamma, c["eps"], c["positions"], c["table"],
                                 w.slot_mapping, cache_ref, block_size=w.block_size,
                                 kv_lora_rank=R, rope_dim=64, kv_is_fp8=fp8,
                                 scale=w.kv_scale, q_pe=q_ref, **kw)
    _check_bf16(_bits(q_pe), q_ref, what="q_pe")
    got = d.cache_numpy()
    if not fp8:
        _check_bf16(got, cache_ref, what="cache")
        # the crafted ties really are ties: 259/256 -> 1 + 2^-6, 511/512 -> 1
        row0 = got.reshape(-1, R + 64)[3]
        assert row0[3] in (0x3F82, 0xBF82)
        return
    nan_ref = _nan_code(cache_ref, fmt)
    assert np.array_equal(nan_ref, _nan_code(got, fmt))
    _check_bf16(np.where(nan_ref, 0, got), np.where(nan_ref, 0, cache_ref), what="fp8 cache")
