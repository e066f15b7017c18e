"""Pins for the split-count rule.

"Triton and MLA: portable attention and multi-head latent attention", Key
files: _compute_num_kv_splits picks the KV split count from max_seq_len / 512,
capped at sm_count * 2; Data flow: batch-invariant mode uses 1 split.  The body
is not printed; the reading is min(ceil(max_seq_len / 512), 2 * sm_count),
at least 1.
"""
import pytest


@pytest.mark.parametrize("L,sms,det,want", [
    (0, 152, False, 1), (1, 152, False, 1), (512, 152, False, 1), (513, 152, False, 2),
    (4096, 152, False, 8), (3585, 152, False, 8), (3584, 152, False, 7),
    (32768, 152, False, 64), (131072, 152, False, 256), (10 ** 6, 152, False, 304),
    (10 ** 6, 4, False, 8), (4096, 152, True, 1), (10 ** 6, 152, True, 1),
])
def test_split_rule(oracle_mod, L, sms, det, want):
    assert oracle_mod.num_kv_splits(L, sms, det) == want
