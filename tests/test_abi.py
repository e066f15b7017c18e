"""The C-ABI library loads, exports every entry point that include/mla.h
declares, and rejects bad arguments on the host before any launch (so these
run without a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

import mla_paged_kv_concat_gb300 as mla
from mla_paged_kv_concat_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "mla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mla_cache_write", "mla_decode", "mla_num_kv_splits",
              "mla_decode_workspace_bytes", "mla_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, name


def _c_to_ctypes(ctype: str):
    """The ctypes class a C parameter or return type of mla.h marshals as."""
    t = ctype.replace("const", "").strip()
    if t == "void":
        return None
    if "*" in t:
        return "pointer"
    return {"int64_t": ctypes.c_int64, "int": ctypes.c_int, "float": ctypes.c_float,
            "size_t": ctypes.c_size_t, "mla_status": ctypes.c_int, "mla_kv_dtype": ctypes.c_int,
            "mla_decode_path": ctypes.c_int}[t]


def _is_pointer(ct) -> bool:
    return ct in (ctypes.c_void_p, ctypes.c_char_p) or (
        isinstance(ct, type) and issubclass(ct, ctypes._Pointer))


def test_binding_signatures_match_the_header_prototypes():
    """Every prototype's return type, parameter count and parameter types
    agree with the ctypes table the binding loads the library with, so a
    parameter added to or moved in the header cannot go unnoticed."""
    text = open(os.path.join(ROOT, "include", "mla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    protos = re.findall(r"([A-Za-z_][\w\s\*]*?)\b(mla_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text)
    assert {name for _, name, _ in protos} == set(_lib.SIGNATURES)
    for ret, name, params in protos:
        restype, argtypes = _lib.SIGNATURES[name]
        want = _c_to_ctypes(ret)
        if want == "pointer":
            assert restype is ctypes.c_char_p, name
        else:
            assert restype is want, name
        plist = [] if params.strip() == "void" else [x.strip() for x in params.split(",")]
        assert len(plist) == len(argtypes), (name, len(plist), len(argtypes))
        for i, (decl, got) in enumerate(zip(plist, argtypes)):
            ctype = re.sub(r"\b\w+\s*$", "", decl).strip()  # drop the parameter name
            want = _c_to_ctypes(ctype)
            if want == "pointer":
                assert _is_pointer(got), (name, i, decl)
            else:
                assert got is want, (name, i, decl, got)


def test_split_rule_and_workspace_size(lib):
    assert mla.mla_num_kv_splits(4096, 152) == 8
    assert mla.mla_num_kv_splits(0, 152) == 1
    assert mla.mla_num_kv_splits(10 ** 7, 152) == 304
    assert mla.mla_decode_workspace_bytes(64, 16, 8, 512) == 64 * 16 * 8 * 513 * 4
    assert mla.mla_decode_workspace_bytes(64, 16, 1, 512) == 0


def test_workspace_size_overflow_is_refused(lib):
    """A workspace size that does not fit a size_t reads as SIZE_MAX, so no
    caller can pass a buffer that large and the no-alloc entry point refuses
    the call before touching its fixed array (nothing is dereferenced)."""
    size_max = (1 << 64) - 1
    big = (2 ** 31 - 1, 128, 65535, 512)
    assert (2 ** 31 - 1) * 128 * 65535 * 513 * 4 > size_max
    assert mla.mla_decode_workspace_bytes(*big) == size_max
    rows, H, S, R = big
    st = lib.mla_decode_noalloc(FAKE, H * 576, 576, rows, H, FAKE, 0, 64, 64, 64 * 576, R, 64,
                                FAKE, 1, 1, FAKE, 1, 0.1, None, S, FAKE, FAKE, None, None)
    assert st == 3  # MLA_ERR_WORKSPACE_TOO_SMALL
    st = lib.mla_decode(FAKE, H * 576, 576, rows, H, FAKE, 0, 64, 64, 64 * 576, R, 64,
                        FAKE, 1, 1, FAKE, 1, 0.1, None, S, FAKE, size_max - 1, FAKE, FAKE,
                        None, None)
    assert st == 3


def test_status_strings(lib):
    for code in range(5):
        assert lib.mla_status_string(code).decode().startswith("MLA_")


FAKE = 1 << 12  # an aligned non-null host address; validation never dereferences


def _decode_args(**over):
    a = dict(q=FAKE, qrs=16 * 576, qhs=576, rows=2, H=16, cache=FAKE, kvd=0, nb=8, bs=64,
             bstride=64 * 576, R=512, P=64, bt=FAKE, bts=4, maxb=4, sl=FAKE, seqs=2,
             scale=0.07, kvs=None, S=2, ws=FAKE, wsb=10 ** 9, o=FAKE, lse=FAKE, err=None,
             stream=None, path=0)
    a.update(over)
    return list(a.values())


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1), (dict(cache=None), 1), (dict(o=None), 1), (dict(lse=None), 1),
    (dict(bt=None), 1), (dict(sl=None), 1),
    (dict(H=0), 1), (dict(H=129), 1), (dict(S=0), 1), (dict(rows=3), 1),
    (dict(R=384), 2), (dict(P=32), 2), (dict(bs=48), 2), (dict(bs=8), 2),
    (dict(bstride=64 * 576 - 8), 1), (dict(q=FAKE + 2), 1), (dict(qhs=500), 1),
    (dict(kvd=1, kvs=None), 1), (dict(kvd=2, kvs=None), 1), (dict(kvd=7), 1),
    (dict(kvd=3), 1), (dict(path=9), 1),
    (dict(wsb=100), 3), (dict(ws=None), 1), (dict(ws=FAKE + 4), 1),
    (dict(bts=2), 1),
])
def test_decode_rejects_bad_arguments(lib, over, code):
    assert lib.mla_decode_ex(*_decode_args(**over)) == code


def _write_args(**over):
    a = dict(kv_c=FAKE, kcs=512, k_pe=FAKE, kps=64, slots=FAKE, T=4, R=512, P=64,
             cache=FAKE, nb=8, bs=64, bstride=64 * 576, kvd=0, scale=None, err=None,
             stream=None)
    a.update(over)
    return list(a.values())


@pytest.mark.parametrize("over,code", [
    (dict(kv_c=None), 1), (dict(slots=None), 1), (dict(cache=None), 1),
    (dict(T=-1), 1), (dict(R=100), 2), (dict(kvd=1, scale=None), 1),
    (dict(kvd=2, scale=None), 1), (dict(kvd=3, scale=FAKE), 1),
    (dict(bstride=100), 1), (dict(cache=FAKE + 8), 1), (dict(kcs=10), 1),
    (dict(nb=0), 1), (dict(bs=0), 1),
])
def test_cache_write_rejects_bad_arguments(lib, over, code):
    assert lib.mla_cache_write(*_write_args(**over)) == code


def test_zero_work_is_ok_without_touching_memory(lib):
    assert lib.mla_cache_write(*_write_args(T=0, kv_c=None, slots=None)) == 0
    assert lib.mla_decode_ex(*_decode_args(rows=0)) == 0


def _lse_merge_args(**over):
    a = dict(o_parts=FAKE, ops=2 * 16 * 512, lse_parts=FAKE, lps=2 * 16, G=3, rows=2, H=16,
             R=512, o=FAKE, lse=FAKE, stream=None)
    a.update(over)
    return list(a.values())


@pytest.mark.parametrize("over,code", [
    (dict(o_parts=None), 1), (dict(lse_parts=None), 1), (dict(o=None), 1), (dict(lse=None), 1),
    (dict(G=0), 1), (dict(G=1025), 1), (dict(H=0), 1), (dict(H=129), 1), (dict(rows=-1), 1),
    (dict(R=384), 2), (dict(ops=2 * 16 * 512 - 8), 1), (dict(ops=2 * 16 * 512 + 4), 1),
    (dict(lps=31), 1), (dict(o_parts=FAKE + 8), 1), (dict(o=FAKE + 8), 1),
    (dict(lse=FAKE + 2), 1),
])
def test_lse_merge_rejects_bad_arguments(lib, over, code):
    assert lib.mla_lse_merge(*_lse_merge_args(**over)) == code


def test_lse_merge_zero_rows_is_a_noop(lib):
    assert lib.mla_lse_merge(*_lse_merge_args(rows=0, o_parts=None, o=None)) == 0


def _nr_args(**over):
    a = dict(kv_c=FAKE, kcs=512, k_pe=FAKE, kps=64, slots=FAKE, T=4, R=512, P=64,
             cache=FAKE, nb=8, bs=64, bstride=64 * 576, kvd=0, scale=None, gamma=FAKE,
             eps=1e-6, pos=FAKE, table=FAKE, maxpos=4096, q_pe=None, qrs=0, qhs=0, qh=0,
             err=None, stream=None)
    a.update(over)
    return list(a.values())


@pytest.mark.parametrize("over,code", [
    (dict(kv_c=None), 1), (dict(gamma=None), 1), (dict(pos=None), 1), (dict(table=None), 1),
    (dict(slots=None), 1), (dict(cache=None), 1), (dict(T=-1), 1), (dict(maxpos=0), 1),
    (dict(eps=-1.0), 1), (dict(eps=float("nan")), 1), (dict(P=32), 2), (dict(R=384), 2),
    (dict(kvd=1, scale=None), 1), (dict(kcs=516), 1), (dict(kv_c=FAKE + 8), 1),
    (dict(gamma=FAKE + 4), 1), (dict(table=FAKE + 4), 1), (dict(bstride=100), 1),
    (dict(q_pe=FAKE, qrs=16 * 64, qhs=64, qh=0), 1),
    (dict(q_pe=FAKE, qrs=16 * 64, qhs=60, qh=16), 1),
    (dict(q_pe=FAKE, qrs=15 * 64, qhs=64, qh=16), 1),
    (dict(q_pe=FAKE + 2, qrs=16 * 64, qhs=64, qh=16), 1),
])
def test_norm_rope_cache_write_rejects_bad_arguments(lib, over, code):
    assert lib.mla_norm_rope_cache_write(*_nr_args(**over)) == code


def test_norm_rope_cache_write_zero_tokens_is_a_noop(lib):
    assert lib.mla_norm_rope_cache_write(*_nr_args(T=0, kv_c=None, slots=None)) == 0


def test_decode_desc_layout_matches_the_header():
    """The ctypes mirror of mla_decode_desc has the C compiler's field offsets."""
    fields = [f for f, _ in _lib.DecodeDesc._fields_]
    src = ['#include <stdio.h>', '#include <stddef.h>', '#include "mla.h"', 'int main(void) {',
           'printf("%zu\\n", sizeof(mla_decode_desc));']
    src += [f'printf("%zu\\n", offsetof(mla_decode_desc, {f}));' for f in fields]
    src += ['return 0; }']
    out = os.path.join(ROOT, "_build", "desc_layout")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    with open(out + ".c", "w") as f:
        f.write("\n".join(src) + "\n")
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), out + ".c", "-o", out],
                   check=True, capture_output=True)
    got = [int(x) for x in subprocess.run([out], check=True, capture_output=True,
                                          text=True).stdout.split()]
    assert got[0] == ctypes.sizeof(_lib.DecodeDesc)
    assert got[1:] == [getattr(_lib.DecodeDesc, f).offset for f in fields]


def test_plan_create_validates_before_anything_runs(lib):
    plan = ctypes.c_void_p(123)
    assert lib.mla_plan_create(None, ctypes.byref(plan)) == 1 and plan.value is None
    d = _lib.DecodeDesc(q=FAKE, q_row_stride=16 * 576, q_head_stride=576, num_rows=2,
                        num_heads=16, kv_cache=FAKE, num_blocks=8, block_size=64,
                        block_stride=64 * 576, kv_lora_rank=512, rope_dim=64, block_table=FAKE,
                        block_table_stride=4, max_blocks_per_seq=4, seq_lens=FAKE, num_seqs=2,
                        sm_scale=0.07, num_kv_splits=1, o=FAKE, lse=FAKE)
    bad = [dict(q=None), dict(num_heads=129), dict(kv_lora_rank=384), dict(q_head_stride=512),
           dict(q_head_stride=512, q_pe=FAKE, q_pe_row_stride=16 * 64, q_pe_head_stride=60),
           dict(q_pe=FAKE + 2, q_head_stride=512, q_pe_row_stride=16 * 64, q_pe_head_stride=64),
           dict(num_tokens=2, kv_c=None, k_pe=FAKE, slot_mapping=FAKE, kv_c_row_stride=512,
                k_pe_row_stride=64),
           dict(num_tokens=3, kv_c=FAKE, k_pe=FAKE, slot_mapping=FAKE, kv_c_row_stride=512,
                k_pe_row_stride=64, gamma=FAKE, positions=FAKE, cos_sin_table=FAKE,
                max_position=100, rotate_q=1),
           dict(num_tokens=-1)]
    for over in bad:
        dd = _lib.DecodeDesc.from_buffer_copy(d)
        for k, v in over.items():
            setattr(dd, k, v)
        plan = ctypes.c_void_p(123)
        st = lib.mla_plan_create(ctypes.byref(dd), ctypes.byref(plan))
        assert st in (1, 2), (over, st)
        assert plan.value is None, over
    assert lib.mla_plan_run(None, None) == 1
    lib.mla_plan_destroy(None)
