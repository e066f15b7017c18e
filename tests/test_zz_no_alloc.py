"""mla_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (for example a plugin whose host application owns every device
allocation through its own pool, or a serving loop that may not call
cudaMalloc / cudaFree because they can block or synchronise the device).

It must give the same results as mla_decode with a caller-allocated
workspace, call after call, while keeping its split partials in the
library's built-in array.  This file is collected last so that a run that
stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import mla_paged_kv_concat_gb300 as mla
from mla_paged_kv_concat_gb300 import workloads as W

from _helpers import Dev, sm_count

pytestmark = pytest.mark.gpu

LIMIT = 32 << 20  # MLA_NOALLOC_WORKSPACE_BYTES in include/mla.h


def _noalloc(lib, d, w, S, o, lse):
    D = w.head_dim
    nb, bs = w.kv_cache.shape[0], w.block_size
    return lib.mla_decode_noalloc(
        d.q.data_ptr(), d.q.stride(0), d.q.stride(1), w.num_rows, w.num_heads,
        d.cache.data_ptr(), mla.MLA_KV_FP8_E4M3 if w.kv_fp8 else mla.MLA_KV_BF16, nb, bs,
        bs * D, w.kv_lora_rank, w.rope_dim, d.block_table.data_ptr(), d.block_table.stride(0),
        d.block_table.shape[1], d.seq_lens.data_ptr(), w.num_seqs, w.sm_scale,
        d.kv_scale.data_ptr(), S, o.data_ptr(), lse.data_ptr(), d.err.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


# Workloads small enough for the built-in array, one per stage-1 kernel and
# cache format: the warp-MMA kernel on bf16 (per_shard, tiny) and on an E4M3
# cache, and the tcgen05 kernel (128 heads).  S = None takes the split rule.
CASES = {
    "per_shard": (None, None),
    "tiny": (None, 2),
    "tcgen05_h128": (dict(seq_lens=[4096] * 12 + [1000, 64, 3000, 70], num_heads=128,
                          pool_blocks=900), 4),
    "fp8_h32": (dict(seq_lens=[512, 4000, 2000, 33, 1500, 4096, 900, 2600], num_heads=32,
                     kv_lora_rank=256, kv_fp8=True, kv_scale=0.05, write="all"), None),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_mla_decode_twice(cuda_dev, name):
    """Same kernels, same partition: the results must be bitwise equal to
    mla_decode's with a caller-allocated workspace, on two calls in a row
    (the second finds the first call's partials in the array)."""
    lib = mla.load()
    kw, S = CASES[name]
    w = W.make(name) if kw is None else W.make_workload(name, seed=91, **kw)
    if S is None:
        S = mla.mla_num_kv_splits(w.max_seq_len, sm_count())
    assert 0 < mla.mla_decode_workspace_bytes(w.num_rows, w.num_heads, S, w.kv_lora_rank) <= LIMIT
    d = Dev(w)
    d.write()
    o_ref, lse_ref = d.decode(S)  # caller-allocated workspace
    o_ref, lse_ref = o_ref.clone(), lse_ref.clone()
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        assert _noalloc(lib, d, w, S, o, lse) == 0
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))
    assert int(d.err.item()) == 0


def test_noalloc_refuses_workspace_beyond_its_array(cuda_dev):
    lib = mla.load()
    w = W.make("tiny")
    d = Dev(w)
    S = 60000  # 2 rows x 16 heads x 60000 splits x 513 x 4 B > 32 MiB
    assert mla.mla_decode_workspace_bytes(w.num_rows, w.num_heads, S, w.kv_lora_rank) > LIMIT
    o = torch.empty(w.num_rows, w.num_heads, w.kv_lora_rank, dtype=torch.bfloat16,
                    device="cuda")
    lse = torch.empty(w.num_rows, w.num_heads, dtype=torch.float32, device="cuda")
    assert _noalloc(lib, d, w, S, o, lse) == 3  # MLA_ERR_WORKSPACE_TOO_SMALL
