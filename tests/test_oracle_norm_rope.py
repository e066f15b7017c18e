"""Pins for the oracle's steps upstream of the cache write: one fp64 -> bf16
rounding, the RMSNorm of the latent (kv_a_layernorm) and the non-NeoX rotary
embedding of k_pe / q_pe ("frozenleaves/vllm compare
v0.11.0...mla_cuda_graphs", vllm/model_executor/models/deepseek_v2.py:
kv_a_layernorm = RMSNorm(kv_lora_rank), rotary_emb = get_rope(...,
is_neox_style=False); the MLA common forward rotates q_pe and k_pe by input
position and then calls concat_and_cache_mla).

Each pin is independent of the oracle's own arithmetic: torch's RNE cast for
fp32 inputs, hand-built fp64 cases where rounding through fp32 first would
give another answer, torch CPU float64 rms_norm, numpy complex128
multiplication, and closed forms.
"""
import numpy as np
import pytest
import torch

import oracle
from mla_paged_kv_concat_gb300 import workloads as W


def _bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------ bf16 rounding
def test_bf16_round_matches_torch_on_fp32_inputs(oracle_mod):
    rng = np.random.default_rng(11)
    u = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    x = x[np.isfinite(x)]
    # plus every tie pattern around a few binades and the subnormal range
    ties = (np.arange(-200, 200, dtype=np.int64)[:, None] * 0 +
            np.array([0x3F808000, 0x3F818000, 0x00008000, 0x00018000, 0x7F7F8000,
                      0x80008000, 0x0001FFFF, 0x3F7FFFFF], np.int64)[None, :])
    x = np.concatenate([x, ties.ravel().astype(np.uint32).view(np.float32)])
    want = _bits_of(torch.from_numpy(x.copy()).to(torch.bfloat16))
    got = oracle.bf16_round(x.astype(np.float64))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("x,bits", [
    (1.0 + 2.0 ** -8, 0x3F80),                    # tie -> even (down)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),                # tie -> even (up)
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),       # above the tie by less than fp32 resolves
    (1.0 + 2.0 ** -8 - 2.0 ** -40, 0x3F80),
    (-(1.0 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
    (2.0 ** -133, 0x0001),                        # smallest subnormal
    (2.0 ** -134, 0x0000),                        # half of it: tie -> 0
    (2.0 ** -134 + 2.0 ** -170, 0x0001),
    (2.0 ** -126 * (1 - 2.0 ** -9), 0x0080),       # rounds up into the normals
    ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),        # largest finite
    (2.0 ** 128 * (1 - 2.0 ** -9), 0x7F80),        # tie above it -> infinity
    (2.0 ** 128 * (1 - 2.0 ** -9) - 2.0 ** 80, 0x7F7F),
    (-0.0, 0x8000), (float("inf"), 0x7F80), (float("-inf"), 0xFF80), (float("nan"), 0x7FC0),
    (1e300, 0x7F80),
])
def test_bf16_round_single_rounding_cases(oracle_mod, x, bits):
    assert int(oracle.bf16_round([x])[0]) == bits


# ------------------------------------------------------------ RMSNorm
@pytest.mark.parametrize("R,eps", [(512, 1e-6), (256, 1e-6), (512, 0.5)])
def test_rms_norm_matches_torch_float64(oracle_mod, R, eps):
    rng = np.random.default_rng(R)
    x = W.randn_bf16(rng, (37, R))
    x[3] = W.bf16_bits_from_f32((rng.standard_normal(R) * 1e-3).astype(np.float32))
    x[5] = W.bf16_bits_from_f32((rng.standard_normal(R) * 300).astype(np.float32))
    g = W.bf16_bits_from_f32((1 + 0.25 * rng.standard_normal(R)).astype(np.float32))
    xv = torch.from_numpy(oracle.bf16_value(x))
    gv = torch.from_numpy(oracle.bf16_value(g))
    ref = torch.nn.functional.rms_norm(xv, (R,), weight=gv, eps=float(np.float32(eps)))
    got = oracle.rms_norm(x, g, float(np.float32(eps)))
    want = oracle.bf16_round(ref.numpy())
    assert np.array_equal(got, want)


def test_rms_norm_closed_forms(oracle_mod):
    R = 512
    one = np.full(R, 0x3F80, np.uint16)
    # a constant row c: mean square c^2, so x / rms = sign(c) exactly when eps = 0
    for c in (0x3F80, 0xC0A0, 0x0123, 0x7F00):
        out = oracle.rms_norm(np.full((1, R), c, np.uint16), one, 0.0)
        assert np.all(out == (0xBF80 if c & 0x8000 else 0x3F80))
    rng = np.random.default_rng(3)
    x = W.randn_bf16(rng, (4, R))
    g = W.bf16_bits_from_f32((1 + 0.25 * rng.standard_normal(R)).astype(np.float32))
    base = oracle.rms_norm(x, g, 0.0)
    for k in (-20, -1, 3, 40):
        scaled = W.bf16_bits_from_f32((oracle.bf16_value(x) * 2.0 ** k).astype(np.float32))
        assert np.array_equal(oracle.rms_norm(scaled, g, 0.0), base)
    # gamma scales the output element by element
    g2 = W.bf16_bits_from_f32((oracle.bf16_value(g) * 4).astype(np.float32))
    assert np.array_equal(oracle.bf16_value(oracle.rms_norm(x, g2, 0.0)),
                          4 * oracle.bf16_value(base))


# ------------------------------------------------------------ rotary
def _table(P, n, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    ang = rng.uniform(-np.pi, np.pi, size=(n, P // 2))
    return (np.concatenate([np.cos(ang), np.sin(ang)], axis=1) * scale).astype(np.float32)


@pytest.mark.parametrize("P,H,scale", [(64, 1, 1.0), (64, 16, 1.0), (32, 3, 1.25)])
def test_rope_matches_complex_multiplication(oracle_mod, P, H, scale):
    n = 50
    rng = np.random.default_rng(P + H)
    tab = _table(P, 200, seed=H, scale=scale)
    pos = rng.integers(0, 200, size=n)
    x = W.randn_bf16(rng, (n, H, P))
    got = x.copy()
    assert oracle.rope_interleaved(got, pos, tab) == 0
    v = oracle.bf16_value(x)
    z = v[..., 0::2] + 1j * v[..., 1::2]                      # pair i = x[2i] + i x[2i+1]
    rot = tab[pos, :P // 2].astype(np.float64) + 1j * tab[pos, P // 2:].astype(np.float64)
    zr = z * rot[:, None, :]
    want = np.empty_like(v)
    want[..., 0::2], want[..., 1::2] = zr.real, zr.imag
    assert np.array_equal(got, oracle.bf16_round(want))


def test_rope_closed_forms(oracle_mod):
    P, H, n = 64, 4, 8
    rng = np.random.default_rng(5)
    x = W.randn_bf16(rng, (n, H, P))
    tab = np.zeros((3, P), np.float32)
    tab[0, :P // 2] = 1.0                     # position 0: identity
    tab[1, P // 2:] = 1.0                     # position 1: a quarter turn
    tab[2] = _table(P, 1, seed=9)[0]          # position 2: a generic angle per pair
    y = x.copy()
    oracle.rope_interleaved(y, np.zeros(n, np.int64), tab)
    assert np.array_equal(y, x)
    y = x.copy()
    oracle.rope_interleaved(y, np.ones(n, np.int64), tab)
    assert np.array_equal(y[..., 0::2], x[..., 1::2] ^ np.uint16(0x8000))
    assert np.array_equal(y[..., 1::2], x[..., 0::2])
    # a rotation then its inverse gives the input back within two bf16 roundings
    inv = tab.copy()
    inv[:, P // 2:] *= -1
    y = x.copy()
    oracle.rope_interleaved(y, np.full(n, 2, np.int64), tab)
    oracle.rope_interleaved(y, np.full(n, 2, np.int64), inv)
    a, b = oracle.bf16_value(y), oracle.bf16_value(x)
    assert np.all(np.abs(a - b) <= 2 * 2.0 ** -8 * (np.abs(b) + np.abs(np.roll(b, 1, -1))
                                                   + np.abs(np.roll(b, -1, -1))) + 1e-30)
    # pair norms are kept by a unit table
    y = x.copy()
    oracle.rope_interleaved(y, np.full(n, 2, np.int64), tab)
    na = oracle.bf16_value(y)[..., 0::2] ** 2 + oracle.bf16_value(y)[..., 1::2] ** 2
    nb = b[..., 0::2] ** 2 + b[..., 1::2] ** 2
    assert np.allclose(na, nb, rtol=2 ** -6, atol=1e-12)


def test_rope_skips_bad_positions_and_uses_the_row_position(oracle_mod):
    P, H = 64, 2
    tab = _table(P, 10, seed=1)
    rng = np.random.default_rng(6)
    x = W.randn_bf16(rng, (4, H, P))
    y = x.copy()
    assert oracle.rope_interleaved(y, np.array([3, -1, 10, 9]), tab) == 2
    assert np.array_equal(y[1], x[1]) and np.array_equal(y[2], x[2])
    one = x[3:4].copy()
    oracle.rope_interleaved(one, np.array([9]), tab)
    assert np.array_equal(y[3], one[0])


# ------------------------------------------------------------ composition
def test_norm_rope_cache_write_special_cases(oracle_mod):
    w = W.make("tiny")  # 4 written tokens, one of them padded (slot -1)
    x = W.norm_rope_inputs(w, seed=3, num_bad_positions=1)
    pad = int(np.flatnonzero(w.slot_mapping < 0)[0])
    bad = int(np.flatnonzero((x.positions < 0) | (x.positions >= x.table.shape[0]))[0])
    cache = w.kv_cache.copy()
    q_pe = _bits_of(x.q_pe).copy()
    nslot, npos = oracle.norm_rope_cache_write(
        w.kv_c, w.k_pe, x.gamma, x.eps, x.positions, x.table, w.slot_mapping, cache,
        block_size=w.block_size, kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim,
        kv_is_fp8=False, q_pe=q_pe)
    assert nslot == 0 and npos == 1
    q0 = _bits_of(x.q_pe)
    assert np.array_equal(q_pe[bad], q0[bad])                 # bad position: untouched
    if pad != bad:
        assert not np.array_equal(q_pe[pad], q0[pad])         # padded token: still rotated
    bs, D = w.block_size, w.head_dim
    flat = cache.reshape(-1, D)
    before = w.kv_cache.reshape(-1, D)
    for t, s in enumerate(w.slot_mapping):
        if s < 0:
            continue
        if t == bad:
            assert np.array_equal(flat[s], before[s])          # nothing written
            continue
        normed = oracle.rms_norm(_bits_of(w.kv_c)[t:t + 1], _bits_of(x.gamma), x.eps)[0]
        assert np.array_equal(flat[s, :w.kv_lora_rank], normed)
    written = {int(s) for t, s in enumerate(w.slot_mapping) if s >= 0 and t != bad}
    others = np.array([i for i in range(flat.shape[0]) if i not in written])
    assert np.array_equal(flat[others], before[others])
