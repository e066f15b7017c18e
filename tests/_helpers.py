"""Shared helpers for the GPU parity tests: move a workload to the device, run
the library through its C ABI, run the oracle on the same host inputs, and
compare at the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import mla_paged_kv_concat_gb300 as mla
import oracle
from mla_paged_kv_concat_gb300 import workloads as W

# Tolerances for bf16 attention outputs against the fp64 oracle:
#   |o - ref| <= O_ATOL + O_RTOL * |ref|,   |lse - ref| <= LSE_ATOL.
O_ATOL = 1e-2
O_RTOL = 1e-2
LSE_ATOL = 2e-3


class Dev:
    """Device copies of one workload's tensors."""

    def __init__(self, w: W.Workload, device="cuda"):
        self.w = w
        self.q = w.q.to(device)
        if w.kv_fp8:
            self.cache = torch.from_numpy(w.kv_cache.copy()).to(device)
        else:
            self.cache = torch.from_numpy(w.kv_cache.view(np.int16).copy()).view(
                torch.bfloat16).to(device)
        self.block_table = torch.from_numpy(w.block_table).to(device)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(device)
        self.kv_c = w.kv_c.to(device)
        self.k_pe = w.k_pe.to(device)
        self.slot_mapping = torch.from_numpy(w.slot_mapping).to(device)
        self.kv_scale = torch.tensor([w.kv_scale], dtype=torch.float32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def write(self):
        mla.cache_write(self.kv_c, self.k_pe, self.cache, self.slot_mapping,
                        scale=self.kv_scale if self.w.kv_fp8 else None, err_count=self.err)

    def decode(self, num_kv_splits, path=mla.MLA_PATH_AUTO, **kw):
        w = self.w
        return mla.decode(self.q, self.cache, self.block_table, self.seq_lens, w.sm_scale,
                          num_kv_splits, kv_lora_rank=w.kv_lora_rank,
                          kv_scale=self.kv_scale if w.kv_fp8 else None, err_count=self.err,
                          path=path, **kw)

    def cache_numpy(self) -> np.ndarray:
        c = self.cache.cpu()
        if self.w.kv_fp8:
            return c.numpy()
        return c.view(torch.int16).numpy().view(np.uint16)


def oracle_cache(w: W.Workload) -> np.ndarray:
    cache = w.kv_cache.copy()
    oracle.cache_write(w.kv_c, w.k_pe, w.slot_mapping, cache, block_size=w.block_size,
                       kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim, kv_is_fp8=w.kv_fp8,
                       scale=w.kv_scale)
    return cache


def oracle_decode(w: W.Workload, cache: np.ndarray, pairs=None, splits: int = 0):
    return oracle.decode(w.q, cache, w.block_table, w.seq_lens, block_size=w.block_size,
                         kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim,
                         sm_scale=w.sm_scale, kv_is_fp8=w.kv_fp8, kv_scale=w.kv_scale,
                         num_kv_splits=splits, pairs=pairs)


def sample_pairs(w: W.Workload, n: int, seed: int = 0) -> np.ndarray:
    """n distinct (row, head) pairs, always including the first and last."""
    total = w.num_rows * w.num_heads
    rng = np.random.default_rng(seed)
    idx = np.unique(np.concatenate([[0, total - 1], rng.choice(total, size=min(n, total),
                                                               replace=False)]))
    return np.stack([idx // w.num_heads, idx % w.num_heads], axis=1)


def unit_pairs(w: W.Workload, unit: int, extra: int = 0, seed: int = 0) -> np.ndarray:
    """(row, head) pairs that reach every unit of a stage-1 schedule: the
    first and last query vector of each `unit`-vector block of each sequence
    (a sequence's rows_per_seq * H vectors in row-major order), plus `extra`
    random pairs."""
    H = w.num_heads
    nvec = w.rows_per_seq * H
    flat = []
    for b in range(w.num_seqs):
        for g0 in range(0, nvec, unit):
            for v in (g0, min(g0 + unit, nvec) - 1):
                flat.append((b * w.rows_per_seq + v // H) * H + v % H)
    if extra:
        rng = np.random.default_rng(seed)
        flat.extend(rng.choice(w.num_rows * H, size=min(extra, w.num_rows * H),
                               replace=False).tolist())
    idx = np.unique(np.asarray(flat, np.int64))
    return np.stack([idx // H, idx % H], axis=1)


def assert_close(o_gpu: torch.Tensor, lse_gpu: torch.Tensor, o_ref: np.ndarray,
                 lse_ref: np.ndarray, pairs=None, what=""):
    R = o_ref.shape[-1]
    og = o_gpu.float().cpu().numpy().astype(np.float64).reshape(-1, R)
    lg = lse_gpu.cpu().numpy().astype(np.float64).reshape(-1)
    if pairs is not None:
        H = o_gpu.shape[1]
        flat = pairs[:, 0] * H + pairs[:, 1]
        og, lg = og[flat], lg[flat]
    assert og.shape == o_ref.shape, (og.shape, o_ref.shape)
    err = np.abs(og - o_ref)
    bound = O_ATOL + O_RTOL * np.abs(o_ref)
    bad = ~(err <= bound)
    assert not bad.any(), (
        f"{what}: o mismatch at {np.argwhere(bad)[:5].tolist()} "
        f"max err {np.nanmax(err):.3e}; gpu {og[bad][:5]} ref {o_ref[bad][:5]}")
    both_inf = np.isneginf(lg) & np.isneginf(lse_ref)
    lerr = np.where(both_inf, 0.0, np.abs(lg - lse_ref))
    badl = ~(lerr <= LSE_ATOL)
    assert not badl.any(), (
        f"{what}: lse mismatch at {np.argwhere(badl)[:5].ravel().tolist()} "
        f"gpu {lg[badl][:5]} ref {lse_ref[badl][:5]}")
    return float(np.nanmax(err)) if err.size else 0.0, float(np.nanmax(lerr)) if lerr.size else 0.0


def sm_count() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count
