"""ctypes view of libmla.so: the C ABI declared in include/mla.h, same names.

Argument marshalling only; every step of the computation runs in the CUDA
kernels behind these symbols.  Loading fails loudly when the library has not
been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE_TOO_SMALL = 3
MLA_ERR_CUDA = 4

MLA_KV_BF16 = 0
MLA_KV_FP8_E4M3 = 1
MLA_KV_FP8_E5M2 = 2

MLA_PATH_AUTO = 0
MLA_PATH_MMA_SYNC = 1
MLA_PATH_TCGEN05 = 2



class DecodeDesc(ctypes.Structure):
    """mla_decode_desc (include/mla.h), field for field."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("q_row_stride", ctypes.c_int64),
        ("q_head_stride", ctypes.c_int64),
        ("q_pe", ctypes.c_void_p), ("q_pe_row_stride", ctypes.c_int64),
        ("q_pe_head_stride", ctypes.c_int64),
        ("num_rows", ctypes.c_int), ("num_heads", ctypes.c_int),
        ("kv_cache", ctypes.c_void_p), ("kv_dtype", ctypes.c_int),
        ("num_blocks", ctypes.c_int), ("block_size", ctypes.c_int),
        ("block_stride", ctypes.c_int64),
        ("kv_lora_rank", ctypes.c_int), ("rope_dim", ctypes.c_int),
        ("kv_scale", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("block_table_stride", ctypes.c_int64),
        ("max_blocks_per_seq", ctypes.c_int),
        ("seq_lens", ctypes.c_void_p), ("num_seqs", ctypes.c_int),
        ("sm_scale", ctypes.c_float), ("num_kv_splits", ctypes.c_int),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("err_count", ctypes.c_void_p),
        ("path", ctypes.c_int),
        ("kv_c", ctypes.c_void_p), ("kv_c_row_stride", ctypes.c_int64),
        ("k_pe", ctypes.c_void_p), ("k_pe_row_stride", ctypes.c_int64),
        ("slot_mapping", ctypes.c_void_p), ("num_tokens", ctypes.c_int),
        ("gamma", ctypes.c_void_p), ("eps", ctypes.c_float),
        ("positions", ctypes.c_void_p), ("cos_sin_table", ctypes.c_void_p),
        ("max_position", ctypes.c_int64), ("rotate_q", ctypes.c_int),
    ]


# Every exported symbol and its (restype, argtypes).
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int
_F32 = ctypes.c_float
_SZ = ctypes.c_size_t
SIGNATURES = {
    "mla_cache_write": (_I32, [_P, _I64, _P, _I64, _P, _I32, _I32, _I32, _P, _I32, _I32,
                               _I64, _I32, _P, _P, _P]),
    "mla_num_kv_splits": (_I32, [_I64, _I32]),
    "mla_decode_workspace_bytes": (_SZ, [_I32, _I32, _I32, _I32]),
    "mla_decode": (_I32, [_P, _I64, _I64, _I32, _I32, _P, _I32, _I32, _I32, _I64, _I32, _I32,
                          _P, _I64, _I32, _P, _I32, _F32, _P, _I32, _P, _SZ, _P, _P, _P, _P]),
    "mla_decode_ex": (_I32, [_P, _I64, _I64, _I32, _I32, _P, _I32, _I32, _I32, _I64, _I32,
                             _I32, _P, _I64, _I32, _P, _I32, _F32, _P, _I32, _P, _SZ, _P, _P,
                             _P, _P, _I32]),
    "mla_decode_splitkv": (_I32, [_P, _I64, _I64, _I32, _I32, _P, _I32, _I32, _I32, _I64,
                                  _I32, _I32, _P, _I64, _I32, _P, _I32, _F32, _P, _I32, _P,
                                  _SZ, _P, _P, _P, _P, _I32]),
    "mla_decode_merge": (_I32, [_I32, _I32, _I32, _P, _I32, _I32, _I32, _I32, _P, _SZ, _P, _P,
                                _P]),
    "mla_decode_noalloc": (_I32, [_P, _I64, _I64, _I32, _I32, _P, _I32, _I32, _I32, _I64,
                                  _I32, _I32, _P, _I64, _I32, _P, _I32, _F32, _P, _I32, _P,
                                  _P, _P, _P]),
    "mla_norm_rope_cache_write": (_I32, [_P, _I64, _P, _I64, _P, _I32, _I32, _I32, _P, _I32,
                                         _I32, _I64, _I32, _P, _P, _F32, _P, _P, _I64, _P,
                                         _I64, _I64, _I32, _P, _P]),
    "mla_lse_merge": (_I32, [_P, _I64, _P, _I64, _I32, _I32, _I32, _I32, _P, _P, _P]),
    "mla_plan_create": (_I32, [ctypes.POINTER(DecodeDesc), ctypes.POINTER(ctypes.c_void_p)]),
    "mla_plan_run": (_I32, [_P, _P]),
    "mla_plan_destroy": (None, [_P]),
    "mla_status_string": (ctypes.c_char_p, [_I32]),
    "mla_last_cuda_error": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        msg = lib.mla_status_string(status).decode()
        if status == MLA_ERR_CUDA:
            msg += ": " + lib.mla_last_cuda_error().decode()
        super().__init__(f"{where}: {msg}")
        self.status = status


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libmla.so (built by ``mla_paged_kv_concat_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(
                f"libmla.so not found at {p}: build it with "
                "`python -m mla_paged_kv_concat_gb300.build` (no CPU fallback exists)")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def check(status: int, where: str) -> None:
    if status != MLA_OK:
        raise MlaError(status, where)
