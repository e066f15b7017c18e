"""MLA decode over a paged latent KV cache, GB300-native (sm_103a).

Thin Python binding over the C ABI of ``libmla.so`` (``include/mla.h``):

* ``mla_cache_write``, ``mla_decode``, ``mla_decode_ex``,
  ``mla_num_kv_splits``, ``mla_decode_workspace_bytes`` — the C entry points
  under the same names, taking raw device pointers (ints) and a stream handle.
* ``mla_norm_rope_cache_write`` and ``norm_rope_cache_write(...)`` — the cache
  write fused with the RMSNorm of kv_c and the rotary embedding of k_pe / q_pe.
* ``DecodePlan`` — ``mla_plan_create`` / ``mla_plan_run``: a validated step
  over fixed tensors whose ``run()`` only launches kernels (CUDA-graph safe).
* ``mla_lse_merge`` and ``lse_merge(...)`` — the cross-shard LSE merge of
  per-shard (o, lse) pairs (decode context parallelism).
* ``cache_write(...)`` and ``decode(...)`` — torch-tensor conveniences that
  only marshal pointers, strides and the current CUDA stream; every step of
  the computation runs in the library's CUDA kernels.

PyTorch supplies device memory and streams; nothing here computes the method.
"""
from __future__ import annotations

from . import _lib
from ._lib import (MLA_KV_BF16, MLA_KV_FP8_E4M3, MLA_KV_FP8_E5M2, MLA_PATH_AUTO,
                   MLA_PATH_MMA_SYNC, MLA_PATH_TCGEN05, MlaError, load)

__all__ = [
    "mla_cache_write", "mla_decode", "mla_decode_ex", "mla_num_kv_splits",
    "mla_decode_workspace_bytes", "mla_lse_merge", "mla_norm_rope_cache_write",
    "cache_write", "norm_rope_cache_write", "decode", "lse_merge", "DecodePlan",
    "MlaError", "load",
    "MLA_KV_BF16", "MLA_KV_FP8_E4M3", "MLA_KV_FP8_E5M2", "MLA_PATH_AUTO", "MLA_PATH_MMA_SYNC",
    "MLA_PATH_TCGEN05",
]


# ---------------------------------------------------------------- raw C ABI
def mla_cache_write(*args) -> int:
    return load().mla_cache_write(*args)


def mla_decode(*args) -> int:
    return load().mla_decode(*args)


def mla_decode_ex(*args) -> int:
    return load().mla_decode_ex(*args)


def mla_norm_rope_cache_write(*args) -> int:
    return load().mla_norm_rope_cache_write(*args)


def mla_lse_merge(*args) -> int:
    return load().mla_lse_merge(*args)


def mla_num_kv_splits(max_seq_len: int, sm_count: int) -> int:
    return int(load().mla_num_kv_splits(int(max_seq_len), int(sm_count)))


def mla_decode_workspace_bytes(num_rows: int, num_heads: int, num_kv_splits: int,
                               kv_lora_rank: int) -> int:
    return int(load().mla_decode_workspace_bytes(num_rows, num_heads, num_kv_splits,
                                                 kv_lora_rank))


# ---------------------------------------------------------------- torch glue
def _torch():
    import torch
    return torch


def _stream_ptr(stream=None) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _kv_dtype(kv_cache, kv_cache_dtype: str | None) -> int:
    torch = _torch()
    if kv_cache_dtype in (None, "auto"):
        if kv_cache.dtype == torch.bfloat16:
            return MLA_KV_BF16
        if kv_cache.dtype in (torch.uint8, torch.float8_e4m3fn):
            return MLA_KV_FP8_E4M3
        if kv_cache.dtype == torch.float8_e5m2:
            return MLA_KV_FP8_E5M2
        raise ValueError(f"unsupported cache dtype {kv_cache.dtype}")
    if kv_cache_dtype in ("fp8", "fp8_e4m3"):
        return MLA_KV_FP8_E4M3
    if kv_cache_dtype == "fp8_e5m2":
        return MLA_KV_FP8_E5M2
    if kv_cache_dtype == "bf16":
        return MLA_KV_BF16
    raise ValueError(f"unsupported kv_cache_dtype {kv_cache_dtype!r}")


def _cache_geom(kv_cache):
    """(num_blocks, block_size, D, block_stride) of a [NB, bs, D] cache view."""
    nb, bs, d = kv_cache.shape
    assert kv_cache.stride(2) == 1 and kv_cache.stride(1) == d, "cache rows must be dense"
    return nb, bs, d, kv_cache.stride(0)


def cache_write(kv_c, k_pe, kv_cache, slot_mapping, kv_cache_dtype: str | None = None,
                scale=None, err_count=None, stream=None) -> None:
    """Write [kv_c | k_pe] rows into ``kv_cache`` at ``slot_mapping`` (in place).

    Same operands as the pages' concat_and_cache_mla(kv_c, k_pe, kv_cache,
    slot_mapping, kv_cache_dtype, scale); ``scale`` is a device fp32 tensor
    (fp8 caches only).
    """
    kvd = _kv_dtype(kv_cache, kv_cache_dtype)
    nb, bs, d, bstride = _cache_geom(kv_cache)
    assert kv_c.stride(1) == 1 and k_pe.stride(1) == 1
    R, P = kv_c.shape[1], k_pe.shape[1]
    assert R + P == d
    st = load().mla_cache_write(
        kv_c.data_ptr(), kv_c.stride(0), k_pe.data_ptr(), k_pe.stride(0),
        slot_mapping.data_ptr(), slot_mapping.numel(), R, P, kv_cache.data_ptr(), nb, bs,
        bstride, kvd, scale.data_ptr() if scale is not None else None,
        err_count.data_ptr() if err_count is not None else None, _stream_ptr(stream))
    _lib.check(st, "mla_cache_write")


def norm_rope_cache_write(kv_c, k_pe, kv_cache, slot_mapping, gamma, eps: float, positions,
                          cos_sin_table, q_pe=None, kv_cache_dtype: str | None = None,
                          scale=None, err_count=None, stream=None) -> None:
    """RMSNorm(kv_c) * gamma and the non-NeoX rotation of k_pe by position,
    written into ``kv_cache`` at ``slot_mapping``; ``q_pe`` [T, H, 64] (bf16,
    may be the rope columns of q) is rotated in place when given.

    ``gamma`` bf16 [R]; ``positions`` int64 [T]; ``cos_sin_table`` fp32
    [max_position, 64] (cos | sin); ``scale`` a device fp32 tensor (fp8
    caches only).
    """
    kvd = _kv_dtype(kv_cache, kv_cache_dtype)
    nb, bs, d, bstride = _cache_geom(kv_cache)
    assert kv_c.stride(1) == 1 and k_pe.stride(1) == 1 and cos_sin_table.stride(1) == 1
    R, P = kv_c.shape[1], k_pe.shape[1]
    assert R + P == d and cos_sin_table.shape[1] == P
    if q_pe is not None:
        assert q_pe.stride(2) == 1 and q_pe.shape[0] >= slot_mapping.numel()
    st = load().mla_norm_rope_cache_write(
        kv_c.data_ptr(), kv_c.stride(0), k_pe.data_ptr(), k_pe.stride(0),
        slot_mapping.data_ptr(), slot_mapping.numel(), R, P, kv_cache.data_ptr(), nb, bs,
        bstride, kvd, scale.data_ptr() if scale is not None else None, gamma.data_ptr(),
        float(eps), positions.data_ptr(), cos_sin_table.data_ptr(), cos_sin_table.shape[0],
        q_pe.data_ptr() if q_pe is not None else None,
        q_pe.stride(0) if q_pe is not None else 0, q_pe.stride(1) if q_pe is not None else 0,
        q_pe.shape[1] if q_pe is not None else 0,
        err_count.data_ptr() if err_count is not None else None, _stream_ptr(stream))
    _lib.check(st, "mla_norm_rope_cache_write")


def decode(q, kv_cache, block_table, seq_lens, sm_scale: float, num_kv_splits: int, *,
           kv_lora_rank: int | None = None, kv_cache_dtype: str | None = None,
           kv_scale=None, workspace=None, out=None, lse=None, err_count=None,
           stream=None, path: int = MLA_PATH_AUTO):
    """MLA decode; returns (o [rows, H, R] bf16, lse [rows, H] fp32).

    ``q`` [rows, H, R+P] bf16, or the pair (q_nope [rows, H, R], q_pe
    [rows, H, P]) read in place without a concatenation; rows =
    len(seq_lens) * rows_per_seq.  ``kv_cache`` [NB, bs, R+P];
    ``block_table`` int32 [seqs, max_blocks]; ``seq_lens`` int32 [seqs];
    ``kv_scale`` device fp32 tensor for fp8 caches; ``workspace`` a device
    buffer of at least ``mla_decode_workspace_bytes`` bytes (allocated here
    when omitted and needed).
    """
    if isinstance(q, (tuple, list)):
        q_nope, q_pe = q
        plan = DecodePlan(q_nope, kv_cache, block_table, seq_lens, sm_scale, num_kv_splits,
                          q_pe=q_pe, kv_cache_dtype=kv_cache_dtype, kv_scale=kv_scale,
                          workspace=workspace, out=out, lse=lse, err_count=err_count,
                          path=path)
        try:
            plan.run(stream)
        finally:
            plan.close()
        return plan.out, plan.lse
    torch = _torch()
    kvd = _kv_dtype(kv_cache, kv_cache_dtype)
    nb, bs, d, bstride = _cache_geom(kv_cache)
    rows, H, dq = q.shape
    assert dq == d and q.stride(2) == 1
    R = kv_lora_rank if kv_lora_rank is not None else d - 64
    P = d - R
    seqs = seq_lens.numel()
    if out is None:
        out = torch.empty(rows, H, R, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(rows, H, dtype=torch.float32, device=q.device)
    need = mla_decode_workspace_bytes(rows, H, num_kv_splits, R)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().mla_decode_ex(
        q.data_ptr(), q.stride(0), q.stride(1), rows, H, kv_cache.data_ptr(), kvd, nb, bs,
        bstride, R, P, block_table.data_ptr(), block_table.stride(0), block_table.shape[1],
        seq_lens.data_ptr(), seqs, float(sm_scale),
        kv_scale.data_ptr() if kv_scale is not None else None, int(num_kv_splits), ws_ptr,
        ws_bytes, out.data_ptr(), lse.data_ptr(),
        err_count.data_ptr() if err_count is not None else None, _stream_ptr(stream),
        int(path))
    _lib.check(st, "mla_decode")
    return out, lse


class DecodePlan:
    """A validated, prepared decode step over fixed tensors (``mla_plan_*``).

    ``run()`` only launches kernels, so it can be captured into a CUDA graph
    and replayed after new values are copied into the same tensors.  The
    tensors are kept referenced for the plan's life.

    ``q``: [rows, H, R+P] bf16, or dims [0, R) when ``q_pe`` [rows, H, P] is
    given.  ``write``: optional dict(kv_c, k_pe, slot_mapping) of the step's
    new tokens, written before stage 1; ``norm_rope``: optional dict(gamma,
    eps, positions, cos_sin_table, rotate_q) that makes that write the fused
    RMSNorm + rotary write (rotate_q also rotates the query's rope dims in
    place).
    """

    def __init__(self, q, kv_cache, block_table, seq_lens, sm_scale: float, num_kv_splits: int,
                 *, q_pe=None, kv_cache_dtype: str | None = None, kv_scale=None,
                 workspace=None, out=None, lse=None, err_count=None,
                 path: int = MLA_PATH_AUTO, write=None, norm_rope=None):
        import ctypes
        torch = _torch()
        kvd = _kv_dtype(kv_cache, kv_cache_dtype)
        nb, bs, d, bstride = _cache_geom(kv_cache)
        rows, H, dq = q.shape
        assert q.stride(2) == 1
        if q_pe is not None:
            R, P = dq, q_pe.shape[2]
            assert q_pe.shape[:2] == (rows, H) and q_pe.stride(2) == 1
        else:
            R, P = d - 64, 64
            assert dq == d
        assert R + P == d
        if out is None:
            out = torch.empty(rows, H, R, dtype=torch.bfloat16, device=q.device)
        if lse is None:
            lse = torch.empty(rows, H, dtype=torch.float32, device=q.device)
        need = mla_decode_workspace_bytes(rows, H, num_kv_splits, R)
        if need and workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        self.out, self.lse = out, lse
        self._keep = [q, q_pe, kv_cache, block_table, seq_lens, kv_scale, workspace, out, lse,
                      err_count, write, norm_rope]
        ptr = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
        dd = _lib.DecodeDesc(
            q=q.data_ptr(), q_row_stride=q.stride(0), q_head_stride=q.stride(1),
            q_pe=ptr(q_pe), q_pe_row_stride=q_pe.stride(0) if q_pe is not None else 0,
            q_pe_head_stride=q_pe.stride(1) if q_pe is not None else 0,
            num_rows=rows, num_heads=H, kv_cache=kv_cache.data_ptr(), kv_dtype=kvd,
            num_blocks=nb, block_size=bs, block_stride=bstride, kv_lora_rank=R, rope_dim=P,
            kv_scale=ptr(kv_scale), block_table=block_table.data_ptr(),
            block_table_stride=block_table.stride(0), max_blocks_per_seq=block_table.shape[1],
            seq_lens=seq_lens.data_ptr(), num_seqs=seq_lens.numel(), sm_scale=float(sm_scale),
            num_kv_splits=int(num_kv_splits), workspace=ptr(workspace),
            workspace_bytes=workspace.numel() * workspace.element_size()
            if workspace is not None else 0,
            o=out.data_ptr(), lse=lse.data_ptr(), err_count=ptr(err_count), path=int(path))
        if write is not None:
            kv_c, k_pe, slots = write["kv_c"], write["k_pe"], write["slot_mapping"]
            assert kv_c.stride(1) == 1 and k_pe.stride(1) == 1
            dd.kv_c, dd.kv_c_row_stride = kv_c.data_ptr(), kv_c.stride(0)
            dd.k_pe, dd.k_pe_row_stride = k_pe.data_ptr(), k_pe.stride(0)
            dd.slot_mapping, dd.num_tokens = slots.data_ptr(), slots.numel()
            if norm_rope is not None:
                tab = norm_rope["cos_sin_table"]
                assert tab.stride(1) == 1 and tab.shape[1] == P
                dd.gamma = norm_rope["gamma"].data_ptr()
                dd.eps = float(norm_rope["eps"])
                dd.positions = norm_rope["positions"].data_ptr()
                dd.cos_sin_table, dd.max_position = tab.data_ptr(), tab.shape[0]
                dd.rotate_q = int(bool(norm_rope.get("rotate_q", False)))
        handle = ctypes.c_void_p()
        _lib.check(load().mla_plan_create(ctypes.byref(dd), ctypes.byref(handle)),
                   "mla_plan_create")
        self._handle = handle.value

    def run(self, stream=None):
        """Launch the step on ``stream`` (default: the current torch stream)."""
        assert self._handle is not None, "plan closed"
        _lib.check(load().mla_plan_run(self._handle, _stream_ptr(stream)), "mla_plan_run")
        return self.out, self.lse

    def close(self):
        if getattr(self, "_handle", None) is not None:
            load().mla_plan_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def lse_merge(o_parts, lse_parts, *, out=None, lse=None, stream=None):
    """Cross-shard LSE merge; returns (o [rows, H, R] bf16, lse [rows, H] fp32).

    ``o_parts`` bf16 [G, rows, H, R] and ``lse_parts`` fp32 [G, rows, H]: the
    (o, lse) of G disjoint KV token shards of the same query vectors, each
    part dense in (rows, H, R) / (rows, H); lse = -inf marks an empty part.
    """
    torch = _torch()
    G, rows, H, R = o_parts.shape
    assert lse_parts.shape == (G, rows, H)
    assert o_parts.stride()[1:] == (H * R, R, 1) and lse_parts.stride()[1:] == (H, 1)
    if out is None:
        out = torch.empty(rows, H, R, dtype=torch.bfloat16, device=o_parts.device)
    if lse is None:
        lse = torch.empty(rows, H, dtype=torch.float32, device=o_parts.device)
    st = load().mla_lse_merge(
        o_parts.data_ptr(), o_parts.stride(0), lse_parts.data_ptr(), lse_parts.stride(0), G,
        rows, H, R, out.data_ptr(), lse.data_ptr(), _stream_ptr(stream))
    _lib.check(st, "mla_lse_merge")
    return out, lse
