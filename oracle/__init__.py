"""Plain CPU oracle for MLA decode over a paged latent KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (``mla_paged_kv_concat_gb300``) never imports it and
shares no code with it.

The arithmetic lives in ``mla_oracle.c`` (fp64, plain loops, one function per
step, each citing the page passage it restates).  This module only builds that
file with gcc and marshals numpy arrays into it.

Parity status per function (what pins each one is in ``tests/test_oracle_*.py``):

* ``e4m3_value``     pinned: the 256 codes against the OCP E4M3 definition's
                     printed landmarks and torch's float8_e4m3fn -> float.
* ``e4m3_encode``    pinned: all 65,536 bf16 patterns (raw and divided by the
                     fp32 scale 0.05) against torch's float8_e4m3fn cast where
                     |y| <= 448, plus listed ties, saturation and NaN.
* ``e5m2_value``     pinned: the 256 codes against torch's float8_e5m2 ->
                     float and the OCP E5M2 landmarks.
* ``e5m2_encode``    pinned: all 65,536 bf16 patterns (raw and divided by the
                     fp32 scales 0.05 and 3.0) against torch's float8_e5m2
                     cast where |y| <= 57344, plus ties, saturation and NaN.
* ``cache_write``    pinned: numpy fancy-index assignment; slot -1 leaves the
                     cache byte-identical.
* ``decode``         pinned: torch CPU float64 scaled_dot_product_attention and
                     logsumexp over the gathered K/V; L = 1 gives v exactly;
                     equal scores give the mean of v and lse = s + ln L;
                     brute-force fsum log-sum-exp; split route == direct route.
* ``bf16_round``     pinned: every fp32 input against torch's RNE float ->
                     bfloat16 cast (a single rounding there), and fp64 inputs
                     where rounding through fp32 first would differ (listed
                     ties, sticky bits below fp32, subnormals, overflow).
* ``rms_norm``       pinned: torch CPU float64 ``rms_norm`` then one rounding;
                     closed forms (constant rows give +-gamma exactly with
                     eps = 0; power-of-two scaling leaves the output unchanged).
* ``rope_interleaved`` pinned: numpy complex128 multiplication of the
                     interleaved pairs by cos + i sin; cos = 1, sin = 0 is the
                     identity and cos = 0, sin = 1 maps (a, b) to (-b, a)
                     exactly; a rotation and its inverse restore the input.
* ``norm_rope_cache_write`` composes the three with ``cache_write``; pinned
                     by its special cases (padded slots rotate q_pe but write
                     nothing; rows with a position outside the table are left
                     untouched and counted).
* ``num_kv_splits``  pinned: the rule's closed form at the cap, the floor and
                     the 512-token steps.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``mla_oracle.c`` into ``liboracle.so`` (OpenMP when gcc has it)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
        lib.oracle_e4m3_encode_n.argtypes = [P, P, i64]
        lib.oracle_e4m3_value_n.argtypes = [P, P, i64]
        lib.oracle_bf16_value_n.argtypes = [P, P, i64]
        lib.oracle_bf16_round_n.argtypes = [P, P, i64]
        lib.oracle_e5m2_encode_n.argtypes = [P, P, i64]
        lib.oracle_e5m2_value_n.argtypes = [P, P, i64]
        lib.oracle_rms_norm.argtypes = [P, i64, i64, i32, P, ctypes.c_double, P]
        lib.oracle_rms_norm.restype = None
        lib.oracle_rope_interleaved.argtypes = [P, i64, i64, i64, i32, i32, P, P, i64]
        lib.oracle_rope_interleaved.restype = i64
        lib.oracle_cache_write.argtypes = [P, i64, P, i64, P, i64, i32, i32, P,
                                           i64, i32, i64, i32, f32]
        lib.oracle_cache_write.restype = i64
        lib.oracle_decode.argtypes = [P, i64, i64, i32, i32, P, i32, i64, i32,
                                      i64, i32, i32, P, i64, P, i32, f32, f32,
                                      i32, P, i64, P, P, P, i64, P, i32]
        lib.oracle_decode.restype = None
        lib.oracle_num_kv_splits.argtypes = [i64, i32, i32]
        lib.oracle_num_kv_splits.restype = i32
        lib.oracle_max_threads.restype = i32
        lib.oracle_lse_merge.argtypes = [P, P, i32, i64, i32, P, P]
        lib.oracle_lse_merge.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _bits16(a) -> np.ndarray:
    """bf16 data as a uint16 numpy array (accepts torch bf16 or uint16)."""
    if hasattr(a, "view") and hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch  # local: only needed for torch inputs
        return a.contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.asarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def bf16_value(bits) -> np.ndarray:
    b = np.ascontiguousarray(_bits16(bits))
    out = np.empty(b.shape, np.float64)
    _load().oracle_bf16_value_n(_ptr(b), _ptr(out), b.size)
    return out


def e4m3_value(codes) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, np.float64)
    _load().oracle_e4m3_value_n(_ptr(c), _ptr(out), c.size)
    return out


def e4m3_encode(y) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(y, dtype=np.float32))
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e4m3_encode_n(_ptr(v), _ptr(out), v.size)
    return out


def bf16_round(x) -> np.ndarray:
    """fp64 -> bf16 bits, one rounding to nearest even."""
    v = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(v.shape, np.uint16)
    _load().oracle_bf16_round_n(_ptr(v), _ptr(out), v.size)
    return out


def rms_norm(x, gamma, eps: float) -> np.ndarray:
    """RMSNorm of bf16 rows ``x`` [n, R] with bf16 weight ``gamma`` [R];
    returns bf16 bits [n, R]."""
    xb, gb = _bits16(x), np.ascontiguousarray(_bits16(gamma))
    assert xb.ndim == 2 and xb.strides[1] == 2
    n, R = xb.shape
    assert gb.shape == (R,)
    out = np.empty((n, R), np.uint16)
    _load().oracle_rms_norm(_ptr(xb), xb.strides[0] // 2, n, R, _ptr(gb), float(eps), _ptr(out))
    return out


def rope_interleaved(x: np.ndarray, positions, table) -> int:
    """Rotate bf16 bits ``x`` [n, H, P] (uint16, last dim contiguous) in place by
    ``positions`` [n] with the fp32 table [max_position, P] (cos | sin).
    Returns the number of rows skipped for an out-of-range position."""
    assert x.dtype == np.uint16 and x.ndim == 3 and x.strides[2] == 2
    n, H, P = x.shape
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
    tab = np.ascontiguousarray(np.asarray(table, dtype=np.float32))
    assert pos.shape == (n,) and tab.ndim == 2 and tab.shape[1] == P
    return int(_load().oracle_rope_interleaved(_ptr(x), x.strides[0] // 2, x.strides[1] // 2,
                                               n, H, P, _ptr(pos), _ptr(tab), tab.shape[0]))


def norm_rope_cache_write(kv_c, k_pe, gamma, eps: float, positions, table, slot_mapping,
                          kv_cache: np.ndarray, *, block_size: int, kv_lora_rank: int,
                          rope_dim: int, kv_is_fp8: bool, scale: float = 1.0, q_pe=None,
                          fp8_format: str = "e4m3"):
    """RMSNorm of kv_c, rotary embedding of k_pe (and of ``q_pe`` [T, H, P]
    uint16, in place, when given), then the cache write of the results.  A
    token whose position is outside the table is skipped entirely (nothing
    written, its q_pe left as it is).  Returns (skipped slots, skipped
    positions)."""
    kc = _bits16(kv_c)
    T = kc.shape[0]
    normed = rms_norm(kc, gamma, eps)
    rot = np.ascontiguousarray(_bits16(k_pe)[:, None, :rope_dim]).copy()
    bad_pos = rope_interleaved(rot, positions, table)
    if q_pe is not None:
        assert q_pe.shape[0] == T
        rope_interleaved(q_pe, positions, table)
    pos = np.asarray(positions, dtype=np.int64)
    slots = np.asarray(slot_mapping, dtype=np.int64).copy()
    slots[(pos < 0) | (pos >= np.asarray(table).shape[0])] = -1
    bad_slots = cache_write(normed, rot[:, 0, :], slots, kv_cache, block_size=block_size,
                            kv_lora_rank=kv_lora_rank, rope_dim=rope_dim, kv_is_fp8=kv_is_fp8,
                            scale=scale, fp8_format=fp8_format)
    return bad_slots, bad_pos


def e5m2_value(codes) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, np.float64)
    _load().oracle_e5m2_value_n(_ptr(c), _ptr(out), c.size)
    return out


def e5m2_encode(y) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(y, dtype=np.float32))
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e5m2_encode_n(_ptr(v), _ptr(out), v.size)
    return out


def _fp8_kind(kv_is_fp8: bool, fp8_format: str) -> int:
    """0: bf16 cache, 1: E4M3, 2: E5M2 (the C side's kv_is_fp8 argument)."""
    if not kv_is_fp8:
        return 0
    return {"e4m3": 1, "e5m2": 2}[fp8_format]


def num_kv_splits(max_seq_len: int, sm_count: int, deterministic: bool = False) -> int:
    return int(_load().oracle_num_kv_splits(int(max_seq_len), int(sm_count),
                                            int(bool(deterministic))))


def cache_write(kv_c, k_pe, slot_mapping, kv_cache: np.ndarray, *, block_size: int,
                kv_lora_rank: int, rope_dim: int, kv_is_fp8: bool, scale: float = 1.0,
                block_stride: int | None = None, fp8_format: str = "e4m3") -> int:
    """Write tokens into ``kv_cache`` in place; returns the skipped-slot count.

    ``kv_c`` / ``k_pe``: bf16 (torch) or uint16 arrays [T_in, *] whose row
    stride is taken from the array; ``kv_cache``: C-contiguous numpy array
    (uint16 for bf16, uint8 for fp8) whose first axis is the block.
    """
    kc, kp = _bits16(kv_c), _bits16(k_pe)
    assert kc.strides[1] == 2 and kp.strides[1] == 2
    sm = np.ascontiguousarray(np.asarray(slot_mapping, dtype=np.int64))
    assert kv_cache.flags["C_CONTIGUOUS"]
    assert kv_cache.dtype == (np.uint8 if kv_is_fp8 else np.uint16)
    D = kv_lora_rank + rope_dim
    nb = kv_cache.shape[0]
    bstride = block_stride if block_stride is not None else kv_cache.size // nb
    assert bstride >= block_size * D and bstride * nb <= kv_cache.size
    return int(_load().oracle_cache_write(
        _ptr(kc), kc.strides[0] // 2, _ptr(kp), kp.strides[0] // 2, _ptr(sm), sm.size,
        kv_lora_rank, rope_dim, _ptr(kv_cache), nb, block_size, bstride,
        _fp8_kind(kv_is_fp8, fp8_format), float(scale)))


def decode(q, kv_cache: np.ndarray, block_table, seq_lens, *, block_size: int,
           kv_lora_rank: int, rope_dim: int, sm_scale: float, kv_is_fp8: bool = False,
           kv_scale: float = 1.0, num_kv_splits: int = 0, pairs=None,
           block_stride: int | None = None, threads: int | None = None,
           fp8_format: str = "e4m3"):
    """fp64 decode.  Returns (o [n, R] float64, lse [n] float64).

    ``q``: bf16 [rows, H, R+P] (torch or uint16), last dim contiguous.
    ``pairs``: optional int array [n, 2] of (row, head); default all pairs in
    row-major order.  ``num_kv_splits`` 0 = direct definition, >= 1 = the
    split-KV route with its LSE merge.
    """
    qb = _bits16(q)
    assert qb.ndim == 3 and qb.strides[2] == 2
    rows, H, D = qb.shape
    assert D == kv_lora_rank + rope_dim
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    assert bt.ndim == 2 and bt.shape[0] == sl.size and rows % sl.size == 0
    assert kv_cache.flags["C_CONTIGUOUS"]
    nb = kv_cache.shape[0]
    bstride = block_stride if block_stride is not None else kv_cache.size // nb
    maxl = max(int(sl.max()) if sl.size else 1, 1)
    assert maxl <= bt.shape[1] * block_size or int(sl.max()) <= 0
    if pairs is None:
        pr = None
        n = rows * H
    else:
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
        n = pr.shape[0]
    nthr = threads if threads else max_threads()
    o = np.empty((n, kv_lora_rank), np.float64)
    lse = np.empty(n, np.float64)
    ss = np.empty(nthr * maxl, np.float64)
    so = np.empty(nthr * kv_lora_rank, np.float64)
    _load().oracle_decode(
        _ptr(qb), qb.strides[0] // 2, qb.strides[1] // 2, rows, H, _ptr(kv_cache),
        _fp8_kind(kv_is_fp8, fp8_format), nb, block_size, bstride, kv_lora_rank, rope_dim,
        _ptr(bt),
        bt.shape[1], _ptr(sl), sl.size, float(sm_scale), float(kv_scale),
        int(num_kv_splits), None if pr is None else _ptr(pr), n, _ptr(o), _ptr(lse),
        _ptr(ss), maxl, _ptr(so), nthr)
    return o, lse


def lse_merge(o_parts, lse_parts):
    """Cross-shard LSE merge in fp64.  ``o_parts`` [G, n, R], ``lse_parts``
    [G, n] (any float dtype; -inf marks an empty part).  Returns (o [n, R],
    lse [n]) float64."""
    op = np.ascontiguousarray(np.asarray(o_parts, dtype=np.float64))
    lp = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64))
    G, n, R = op.shape
    assert lp.shape == (G, n)
    o = np.empty((n, R), np.float64)
    lse = np.empty(n, np.float64)
    _load().oracle_lse_merge(_ptr(op), _ptr(lp), G, n, R, _ptr(o), _ptr(lse))
    return o, lse
