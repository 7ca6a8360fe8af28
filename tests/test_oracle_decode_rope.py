"""Pins for the oracle's GQA decode and FLUX multi-axis RoPE / joint attention.

Decode: fak "GPU - the in-kernel forward pass" (section 0: device-resident KV
cache; section 4: naive decode attention, one block per head).  GQA grouping
follows Llama's contiguous query-head groups.

RoPE: iris.c issue #15 "CUDA codepath !" (GGML lessons item 3: FLUX's custom
RoPE over 4 axes [32,32,32,32], separate text/image positions,
repeat_interleave) with theta 10000 on adjacent (2i, 2i+1) pairs.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests.brute import dense_attention
from workloads import flux_positions

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- decode --

def test_decode_mha_equals_full_with_one_query():
    B, H, L, D = 2, 3, 40, 32
    q = _rand((B, H, D), 50)
    kc, vc = _rand((B, H, L, D), 51), _rand((B, H, L, D), 52)
    o = oracle.decode_gqa(q, kc, vc, [L, L])
    ref = oracle.full_fwd(q[:, :, None], kc, vc)[:, :, 0]
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-13)


def test_decode_gqa_matches_sdpa_with_repeated_kv_heads():
    B, Hq, Hkv, L, D = 2, 8, 2, 33, 16
    q = _rand((B, Hq, D), 53)
    kc, vc = _rand((B, Hkv, L, D), 54), _rand((B, Hkv, L, D), 55)
    o = oracle.decode_gqa(q, kc, vc, [L, L])
    g = Hq // Hkv
    kr = np.repeat(kc, g, axis=1)      # query head h reads kv head h // g
    vr = np.repeat(vc, g, axis=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q[:, :, None]), torch.from_numpy(kr), torch.from_numpy(vr)).numpy()
    np.testing.assert_allclose(o, ref[:, :, 0], rtol=0, atol=1e-13)


def test_decode_ignores_cache_rows_past_seq_len():
    B, Hq, Hkv, L, D = 3, 4, 1, 50, 8
    q = _rand((B, Hq, D), 56)
    kc, vc = _rand((B, Hkv, L, D), 57), _rand((B, Hkv, L, D), 58)
    sl = [1, 17, 50]
    o = oracle.decode_gqa(q, kc, vc, sl)
    kc2, vc2 = kc.copy(), vc.copy()
    for b, s in enumerate(sl):
        kc2[b, :, s:] = np.nan
        vc2[b, :, s:] = np.nan
    np.testing.assert_array_equal(oracle.decode_gqa(q, kc2, vc2, sl), o)
    # seq_len 1: the output is the first value row
    np.testing.assert_allclose(o[0], np.broadcast_to(vc[0, 0, 0], (Hq, D)), atol=1e-15)
    for b, s in enumerate(sl):
        ref, _ = dense_attention(q[b][:, None], np.repeat(kc[b, :, :s], Hq, 0),
                                 np.repeat(vc[b, :, :s], Hq, 0), 1 / math.sqrt(D))
        np.testing.assert_allclose(o[b], ref[:, 0], rtol=0, atol=1e-13)


# Ring decode (a ring of `capacity` rows keeps the newest tokens; fak section
# 3b names the dynamic / ring device KV as the follow-up to a fixed one).

def _ring_case(seed, B=3, Hq=4, Hkv=2, T=40, D=8):
    g = np.random.default_rng(seed)
    return (g.standard_normal((B, Hq, D)), g.standard_normal((B, Hkv, T, D)),
            g.standard_normal((B, Hkv, T, D)))


def test_ring_decode_one_row_ring_returns_the_newest_value():
    q, kt, vt = _ring_case(60)
    n = [1, 23, 40]
    o = oracle.decode_ring(q, kt, vt, n, capacity=1)
    for b, nb in enumerate(n):
        for h in range(4):
            np.testing.assert_array_equal(o[b, h], vt[b, h // 2, nb - 1])


def test_ring_decode_ignores_tokens_outside_the_window():
    q, kt, vt = _ring_case(61)
    n, cap = [5, 23, 40], 9
    o = oracle.decode_ring(q, kt, vt, n, capacity=cap)
    kt2, vt2 = kt.copy(), vt.copy()
    for b, nb in enumerate(n):
        kt2[b, :, :max(0, nb - cap)] = np.nan     # overwritten by the ring
        vt2[b, :, :max(0, nb - cap)] = np.nan
        kt2[b, :, nb:] = np.nan                   # not yet appended
        vt2[b, :, nb:] = np.nan
    np.testing.assert_array_equal(oracle.decode_ring(q, kt2, vt2, n, capacity=cap), o)


def test_ring_decode_matches_brute_force_on_the_window():
    q, kt, vt = _ring_case(62)
    n, cap = [5, 23, 40], 9
    o = oracle.decode_ring(q, kt, vt, n, capacity=cap)
    for b, nb in enumerate(n):
        lo = max(0, nb - cap)
        kr = np.repeat(kt[b, :, lo:nb], 2, axis=0)    # query head h reads kv head h // 2
        vr = np.repeat(vt[b, :, lo:nb], 2, axis=0)
        ref, _ = dense_attention(q[b][:, None], kr, vr, 1 / math.sqrt(8))
        np.testing.assert_allclose(o[b], ref[:, 0], rtol=0, atol=1e-13)


def test_ring_at_least_as_long_as_the_history_is_plain_decode():
    q, kt, vt = _ring_case(63)
    n = [5, 23, 40]
    np.testing.assert_array_equal(oracle.decode_ring(q, kt, vt, n, capacity=40),
                                  oracle.decode_gqa(q, kt, vt, n))


# ------------------------------------------------------------------ RoPE --

def test_rope_golden_angles():
    g = json.load(open(os.path.join(GOLD, "rope_angles.json")))
    for c in g["cases"]:
        a, i, p = c["axis"], c["pair"], c["pos"]
        pos = np.zeros((1, 4), dtype=np.int32)
        pos[0, a] = p
        ch = 32 * a + 2 * i
        for which, key in ((0, "unit_first"), (1, "unit_second")):
            x = np.zeros((1, 1, 1, 128))
            x[0, 0, 0, ch + which] = 1.0
            y = oracle.rope_rotate(x, pos)[0, 0, 0]
            np.testing.assert_allclose(y[ch:ch + 2], c[key], rtol=0, atol=1e-12)
            rest = np.delete(y, [ch, ch + 1])
            assert np.all(rest == 0)


def test_rope_frequencies_per_axis_block():
    g = json.load(open(os.path.join(GOLD, "rope_angles.json")))
    for i, f in g["freq"].items():
        i = int(i)
        for a in range(4):
            pos = np.zeros((1, 4), dtype=np.int32)
            pos[0, a] = 1
            x = np.zeros((1, 1, 1, 128))
            x[0, 0, 0, 32 * a + 2 * i] = 1.0
            y = oracle.rope_rotate(x, pos)[0, 0, 0]
            assert abs(math.atan2(y[32 * a + 2 * i + 1], y[32 * a + 2 * i]) - f) < 1e-12


def test_rope_identity_at_zero_and_norm_preserving():
    x = _rand((1, 2, 6, 128), 60)
    y0 = oracle.rope_rotate(x, np.zeros((6, 4), dtype=np.int32))
    np.testing.assert_array_equal(y0, x)
    pos = np.random.default_rng(61).integers(0, 600, size=(6, 4)).astype(np.int32)
    y = oracle.rope_rotate(x, pos)
    pair_norm = lambda z: np.sqrt(z[..., 0::2] ** 2 + z[..., 1::2] ** 2)
    np.testing.assert_allclose(pair_norm(y), pair_norm(x), rtol=1e-13, atol=0)


def test_rope_flux_positions_touch_the_right_channels():
    pos = flux_positions(3, 2, 3)
    assert pos.shape == (9, 4)
    x = _rand((1, 1, 9, 128), 62)
    y = oracle.rope_rotate(x, pos)[0, 0]
    # text tokens rotate only channels 96..127 (axis 3); image tokens 32..95
    np.testing.assert_array_equal(y[:3, :96], x[0, 0, :3, :96])
    np.testing.assert_array_equal(y[3:, :32], x[0, 0, 3:, :32])
    np.testing.assert_array_equal(y[3:, 96:], x[0, 0, 3:, 96:])
    assert np.all(y[0] == x[0, 0, 0])          # text token 0 sits at position 0
    assert not np.allclose(y[4, 64:96], x[0, 0, 4, 64:96])   # column 1 rotates axis 2


@pytest.mark.parametrize("axis", [1, 2, 3])
def test_rope_scores_depend_on_relative_position_only(axis):
    N = 12
    q, k = _rand((1, 1, N, 128), 63), _rand((1, 1, N, 128), 64)
    rng = np.random.default_rng(65)
    pos = rng.integers(0, 64, size=(N, 4)).astype(np.int32)
    sh = pos.copy()
    sh[:, axis] += 37
    s1 = oracle.rope_rotate(q, pos)[0, 0] @ oracle.rope_rotate(k, pos)[0, 0].T
    s2 = oracle.rope_rotate(q, sh)[0, 0] @ oracle.rope_rotate(k, sh)[0, 0].T
    np.testing.assert_allclose(s1, s2, rtol=0, atol=1e-11)


def test_joint_equals_full_attention_on_rotated_q_k_only():
    pos = flux_positions(4, 3, 4)
    N = pos.shape[0]
    q, k, v = (_rand((1, 2, N, 128), s) for s in (66, 67, 68))
    o = oracle.joint_fwd(q, k, v, pos)
    qr, kr = oracle.rope_rotate(q, pos), oracle.rope_rotate(k, pos)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qr), torch.from_numpy(kr), torch.from_numpy(v)).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    # all-zero positions reduce to plain attention
    z = np.zeros_like(pos)
    np.testing.assert_allclose(oracle.joint_fwd(q, k, v, z), oracle.full_fwd(q, k, v), atol=1e-14)
    rows = [0, 5, N, 2 * N - 1]
    np.testing.assert_array_equal(oracle.joint_fwd(q, k, v, pos, rows=rows),
                                  o.reshape(-1, 128)[rows])


# -------------------------------------------------------- causal GQA prefill

def test_causal_gqa_matches_sdpa_is_causal_with_repeated_kv():
    B, Hq, Hkv, N, D = 2, 6, 2, 19, 16
    q = _rand((B, Hq, N, D), 70)
    k, v = _rand((B, Hkv, N, D), 71), _rand((B, Hkv, N, D), 72)
    o = oracle.causal_gqa_fwd(q, k, v)
    kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(kr), torch.from_numpy(vr), is_causal=True).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-13)


def test_causal_first_row_is_first_value_and_last_row_is_full_attention():
    B, H, N, D = 1, 2, 11, 8
    q, k, v = (_rand((B, H, N, D), s) for s in (73, 74, 75))
    o = oracle.causal_gqa_fwd(q, k, v)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], atol=1e-15)
    full = oracle.full_fwd(q[:, :, -1:], k, v)
    np.testing.assert_allclose(o[:, :, -1:], full, atol=1e-14)
    # future keys never matter: perturbing them leaves earlier rows unchanged
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 6:] = np.nan
    v2[:, :, 6:] = np.nan
    np.testing.assert_array_equal(oracle.causal_gqa_fwd(q, k2, v2)[:, :, :6], o[:, :, :6])
    rows = [0, 5, 10, 11, 21]
    np.testing.assert_array_equal(oracle.causal_gqa_fwd(q, k, v, rows=rows), o.reshape(-1, D)[rows])
