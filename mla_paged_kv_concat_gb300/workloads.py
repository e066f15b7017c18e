"""Seeded synthetic inputs for MLA decode over a paged latent KV cache.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so the GPU path and the CPU oracle can both consume what
it makes.  Every tensor comes from ``numpy.random.default_rng(PCG64(seed))``,
floats drawn as N(0, 1) fp32 and rounded to bf16 (nearest, ties to even).

The five named workloads restate the DeepSeek-style decode batches that the
benchmark and the tests use:

* ``tiny``        2 sequences, H=16, 512+64, block 64, L = {37, 130}, an 8-block
                  pool (4 used), and a 4-token cache write with one padded slot.
* ``per_shard``   B=64, H=16, 512+64, L ~ U{1024..4096}, 5000-block pool, and a
                  64-token cache write of each sequence's newest token.
* ``full_head``   B=128, H=128, 512+64, L = 4096, 8192-block pool (all used).
* ``fp8_small``   B=32, H=32, 256+64, L log-uniform on [512, 32768]; the fp8
                  cache is written from N(0,1) bf16 tokens with scale 0.05.
* ``long_multirow`` 8 sequences x 4 query rows, H=128, 512+64,
                  L ~ U{65536..131072}, 20000-block pool.

``norm_rope_inputs`` adds, for a workload's written tokens, what the step
upstream of the cache write consumes: the RMSNorm weight, eps, each token's
position and an fp32 cos | sin table of standard rotary frequencies, plus a
q_pe block to rotate.

Memory that the method must never read (blocks outside any sequence, rows past
a sequence's length inside its last block, block-table padding) is filled with
NaN (bf16 0x7FC0, fp8 0x7F), so an unmasked read shows up as NaN.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

BF16_NAN = 0x7FC0
FP8_NAN = 0x7F
SM_SCALE_192 = float(np.float32(1.0 / np.sqrt(192.0)))

WORKLOADS = ("tiny", "per_shard", "full_head", "fp8_small", "long_multirow")


def _rng(seed: int, salt: int) -> np.random.Generator:
    return np.random.default_rng(np.random.PCG64([seed, salt]))


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def randn_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) draws as bf16 bit patterns (uint16)."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    step = 1 << 24
    for i in range(0, n, step):
        m = min(step, n - i)
        out[i:i + m] = bf16_bits_from_f32(rng.standard_normal(m, dtype=np.float32))
    return out.reshape(shape)


def bits_to_torch_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


@dataclass
class Workload:
    """One decode batch plus the cache write that precedes it.

    Shapes: ``q`` [rows, H, R+P] bf16 (torch CPU); ``kv_cache`` [NB, bs, R+P]
    numpy (uint16 bf16 bits, or uint8 e4m3 codes) holding the cache *before*
    the write; ``block_table`` [num_seqs, max_blocks] int32; ``seq_lens``
    [num_seqs] int32; ``kv_c`` [T, R] and ``k_pe`` [T, P] bf16 (torch CPU);
    ``slot_mapping`` [T] int64.
    """
    name: str
    num_seqs: int
    rows_per_seq: int
    num_heads: int
    kv_lora_rank: int
    rope_dim: int
    block_size: int
    kv_fp8: bool
    kv_scale: float
    sm_scale: float
    seq_lens: np.ndarray
    block_table: np.ndarray
    kv_cache: np.ndarray
    q: torch.Tensor
    kv_c: torch.Tensor
    k_pe: torch.Tensor
    slot_mapping: np.ndarray
    meta: dict = field(default_factory=dict)

    @property
    def num_rows(self) -> int:
        return self.num_seqs * self.rows_per_seq

    @property
    def head_dim(self) -> int:
        return self.kv_lora_rank + self.rope_dim

    @property
    def num_blocks(self) -> int:
        return self.kv_cache.shape[0]

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.seq_lens.size else 0

    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_fp8 else 2

    def kv_bytes(self) -> int:
        """Unique latent rows one decode pass must read, in bytes."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.head_dim * self.kv_elem_bytes()

    def flops(self) -> int:
        """2 * H * (R+P + R) per (row, token): the QK^T and PV contractions."""
        per_tok = 2 * self.num_heads * (self.head_dim + self.kv_lora_rank)
        return int(self.seq_lens.astype(np.int64).sum()) * self.rows_per_seq * per_tok


def make_workload(name: str, *, seed: int, seq_lens, num_heads: int, rows_per_seq: int = 1,
                  kv_lora_rank: int = 512, rope_dim: int = 64, block_size: int = 64,
                  pool_blocks: int | None = None, kv_fp8: bool = False, kv_scale: float = 1.0,
                  sm_scale: float = SM_SCALE_192, write: str = "newest",
                  num_write_tokens: int = 0, table_pad: int = 0,
                  poison: bool = True) -> Workload:
    """Build a workload.

    ``write`` chooses the cache write that precedes decode:
      * ``"newest"``: one token per sequence, at slot (L-1) of that sequence
        (its newest token); the cache position is NaN before the write.
      * ``"all"``: every token of every sequence is written (the cache starts
        all-NaN); used for the fp8 cache.
      * ``"random"``: ``num_write_tokens`` tokens at distinct random slots of
        the pool with one padded slot (-1) at a random position.
    ``table_pad`` adds that many padding columns to the block table.
    """
    R, P, bs = kv_lora_rank, rope_dim, block_size
    D = R + P
    sl = np.asarray(seq_lens, dtype=np.int32)
    B = sl.size
    pages = [(int(L) + bs - 1) // bs for L in sl]
    need = int(sum(pages))
    pool = pool_blocks if pool_blocks is not None else need
    assert pool >= need, (pool, need)
    rng_tab = _rng(seed, 1)
    perm = rng_tab.permutation(pool).astype(np.int32)
    maxb = max(max(pages) if pages else 1, 1) + table_pad
    spare = perm[need:]
    pad_id = int(spare[0]) if spare.size else 0
    bt = np.full((B, maxb), pad_id, np.int32)
    k = 0
    for b in range(B):
        bt[b, :pages[b]] = perm[k:k + pages[b]]
        k += pages[b]

    # cache contents before the write
    if kv_fp8:
        cache = np.full((pool, bs, D), FP8_NAN if poison else 0, np.uint8)
    else:
        cache = np.full((pool, bs, D), BF16_NAN if poison else 0, np.uint16)
    rng_kv = _rng(seed, 2)
    if write != "all":
        assert not kv_fp8, "fp8 caches are filled by the cache write"
        for b in range(B):
            L = int(sl[b])
            n_fill = L - 1 if write == "newest" and L > 0 else L
            if n_fill <= 0:
                continue
            vals = randn_bf16(rng_kv, (n_fill, D))
            full, rem = divmod(n_fill, bs)
            for p in range(full):
                cache[bt[b, p]] = vals[p * bs:(p + 1) * bs]
            if rem:
                cache[bt[b, full], :rem] = vals[full * bs:]

    # tokens written before decode
    rng_w = _rng(seed, 3)
    if write == "newest":
        slots = np.array([int(bt[b, (int(sl[b]) - 1) // bs]) * bs + (int(sl[b]) - 1) % bs
                          for b in range(B) if sl[b] > 0], np.int64)
    elif write == "all":
        slots = np.concatenate([
            (bt[b, np.arange(int(sl[b])) // bs].astype(np.int64) * bs + np.arange(int(sl[b])) % bs)
            for b in range(B)]) if B else np.zeros(0, np.int64)
    elif write == "random":
        slots = rng_w.choice(pool * bs, size=num_write_tokens, replace=False).astype(np.int64)
        slots[rng_w.integers(0, num_write_tokens)] = -1
    else:
        raise ValueError(write)
    T = slots.size
    kv_c = bits_to_torch_bf16(randn_bf16(rng_w, (T, R)))
    k_pe = bits_to_torch_bf16(randn_bf16(rng_w, (T, P)))

    rng_q = _rng(seed, 4)
    q = bits_to_torch_bf16(randn_bf16(rng_q, (B * rows_per_seq, num_heads, D)))
    return Workload(name=name, num_seqs=B, rows_per_seq=rows_per_seq, num_heads=num_heads,
                    kv_lora_rank=R, rope_dim=P, block_size=bs, kv_fp8=kv_fp8,
                    kv_scale=float(np.float32(kv_scale)), sm_scale=float(np.float32(sm_scale)),
                    seq_lens=sl, block_table=bt, kv_cache=cache, q=q, kv_c=kv_c, k_pe=k_pe,
                    slot_mapping=slots, meta={"seed": seed, "pool": pool, "write": write})


@dataclass
class NormRopeInputs:
    """Inputs of the RMSNorm + rotary + cache-write step for a workload's T
    written tokens: ``gamma`` bf16 [R] (torch CPU); ``eps`` (an fp32 value);
    ``positions`` int64 [T]; ``table`` fp32 [max_position, P] with cos of
    pair i in column i and sin in column P/2 + i; ``q_pe`` bf16 [T, H, P]
    (torch CPU)."""
    gamma: torch.Tensor
    eps: float
    positions: np.ndarray
    table: np.ndarray
    q_pe: torch.Tensor


def norm_rope_inputs(w: Workload, *, seed: int, max_position: int | None = None,
                     num_bad_positions: int = 0, table_scale: float = 1.0,
                     rope_base: float = 10000.0, q_heads: int | None = None) -> NormRopeInputs:
    """Seeded inputs for the step upstream of the cache write.

    Positions: a sequence's newest token sits at L - 1 (write "newest"),
    every token of a sequence at 0..L-1 (write "all"), otherwise uniform
    over the table.  ``num_bad_positions`` of them are then moved outside
    [0, max_position).  The table holds angles pos * rope_base^(-2i/P)
    (plain rotary frequencies; any fp32 table is a valid input) times
    ``table_scale``.
    """
    R, P = w.kv_lora_rank, w.rope_dim
    T = w.slot_mapping.size
    rng = _rng(seed, 5)
    if max_position is None:
        max_position = max(w.max_seq_len, 1) + 64
    mode = w.meta.get("write")
    if mode == "newest":
        pos = np.array([int(L) - 1 for L in w.seq_lens if L > 0], np.int64)
    elif mode == "all":
        pos = np.concatenate([np.arange(int(L), dtype=np.int64) for L in w.seq_lens]) \
            if w.num_seqs else np.zeros(0, np.int64)
    else:
        pos = rng.integers(0, max_position, size=T).astype(np.int64)
    assert pos.size == T and (T == 0 or pos.max() < max_position)
    if num_bad_positions:
        idx = rng.choice(T, size=num_bad_positions, replace=False)
        pos[idx] = np.where(np.arange(num_bad_positions) % 2 == 0, -1 - idx, max_position + idx)
    inv = rope_base ** (-2.0 * np.arange(P // 2, dtype=np.float64) / P)
    ang = np.arange(max_position, dtype=np.float64)[:, None] * inv[None, :]
    table = (np.concatenate([np.cos(ang), np.sin(ang)], axis=1) * table_scale).astype(np.float32)
    gamma = bf16_bits_from_f32((1.0 + 0.25 * rng.standard_normal(R)).astype(np.float32))
    H = q_heads if q_heads is not None else w.num_heads
    q_pe = randn_bf16(rng, (T, H, P))
    return NormRopeInputs(gamma=bits_to_torch_bf16(gamma), eps=float(np.float32(1e-6)),
                          positions=pos, table=np.ascontiguousarray(table),
                          q_pe=bits_to_torch_bf16(q_pe))


def make(name: str) -> Workload:
    """The five named workloads (seed = 1..5 in the order of ``WORKLOADS``)."""
    if name == "tiny":
        return make_workload(name, seed=1, seq_lens=[37, 130], num_heads=16, pool_blocks=8,
                             write="random", num_write_tokens=4)
    if name == "per_shard":
        sl = _rng(2, 0).integers(1024, 4096, size=64, endpoint=True)
        return make_workload(name, seed=2, seq_lens=sl, num_heads=16, pool_blocks=5000)
    if name == "full_head":
        return make_workload(name, seed=3, seq_lens=[4096] * 128, num_heads=128,
                             pool_blocks=8192)
    if name == "fp8_small":
        u = _rng(4, 0).uniform(np.log(512.0), np.log(32768.0), size=32)
        sl = np.floor(np.exp(u)).astype(np.int64)
        return make_workload(name, seed=4, seq_lens=sl, num_heads=32, kv_lora_rank=256,
                             kv_fp8=True, kv_scale=0.05, write="all")
    if name == "long_multirow":
        sl = _rng(5, 0).integers(65536, 131072, size=8, endpoint=True)
        return make_workload(name, seed=5, seq_lens=sl, num_heads=128, rows_per_seq=4,
                             pool_blocks=20000)
    raise ValueError(name)
