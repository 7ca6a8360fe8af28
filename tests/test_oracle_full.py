"""Pins for the oracle's full (unmasked) attention and the shared softmax core.

Nothing here retypes the oracle's loop: each check is a closed form, a library
routine on a special case, an invariant or an independent dense brute force.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests.brute import dense_attention

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_two_key_closed_form():
    g = json.load(open(os.path.join(GOLD, "two_key_closed_form.json")))
    q = np.array(g["q"])[None, None]
    k = np.array(g["k"])[None, None]
    v = np.array(g["v"])[None, None]
    o, p = oracle.full_fwd(q, k, v, scale=g["scale"], return_p=True)
    np.testing.assert_allclose(p[0, 0, 0], g["p"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(o[0, 0, 0], g["o"], rtol=0, atol=1e-15)


@pytest.mark.parametrize("shape", [(1, 2, 64, 32), (2, 3, 17, 64), (1, 1, 5, 128)])
def test_matches_torch_sdpa_float64(shape):
    B, H, N, D = shape
    q, k, v = (_rand(shape, s) for s in (1, 2, 3))
    o = oracle.full_fwd(q, k, v)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v)).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_rectangular_and_explicit_scale_vs_brute():
    q = _rand((2, 2, 7, 16), 4)
    k = _rand((2, 2, 11, 16), 5)
    v = _rand((2, 2, 11, 16), 6)
    o = oracle.full_fwd(q, k, v, scale=0.3)
    ref, _ = dense_attention(q, k, v, 0.3)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_default_scale_is_inverse_sqrt_d():
    q, k, v = (_rand((1, 1, 9, 32), s) for s in (7, 8, 9))
    np.testing.assert_array_equal(oracle.full_fwd(q, k, v),
                                  oracle.full_fwd(q, k, v, scale=1 / math.sqrt(32)))
    ref, _ = dense_attention(q, k, v, 1 / math.sqrt(32))
    np.testing.assert_allclose(oracle.full_fwd(q, k, v), ref, atol=1e-12)


def test_rows_sum_to_one_and_nonnegative():
    q, k, v = (_rand((1, 2, 33, 32), s) * 3 for s in (10, 11, 12))
    _, p = oracle.full_fwd(q, k, v, return_p=True)
    assert np.all(p >= 0)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)


def test_constant_v_returns_constant():
    q, k = (_rand((1, 2, 20, 32), s) * 4 for s in (13, 14))
    c = _rand((32,), 15)
    v = np.broadcast_to(c, (1, 2, 20, 32)).copy()
    o = oracle.full_fwd(q, k, v)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-12)


def test_zero_q_gives_mean_of_v():
    k, v = (_rand((1, 1, 13, 32), s) for s in (16, 17))
    q = np.zeros((1, 1, 4, 32))
    o = oracle.full_fwd(q, k, v)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0].mean(0), (4, 32)), atol=1e-14)


def test_single_key_returns_its_value():
    q = _rand((1, 1, 3, 8), 18)
    k = _rand((1, 1, 1, 8), 19)
    v = _rand((1, 1, 1, 8), 20)
    o = oracle.full_fwd(q, k, v)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0, 0], (3, 8)), atol=1e-15)


def test_key_permutation_equivariance():
    q, k, v = (_rand((1, 2, 10, 16), s) for s in (21, 22, 23))
    perm = np.random.default_rng(24).permutation(10)
    o1 = oracle.full_fwd(q, k, v)
    o2 = oracle.full_fwd(q, k[:, :, perm], v[:, :, perm])
    np.testing.assert_allclose(o1, o2, atol=1e-14)


def test_large_logits_are_stable():
    # max subtraction: scores of several thousand must not overflow exp
    q, k, v = (_rand((1, 1, 8, 32), s) for s in (25, 26, 27))
    o = oracle.full_fwd(q * 1000, k, v)
    assert np.all(np.isfinite(o))
    s = np.einsum("id,jd->ij", q[0, 0] * 1000, k[0, 0]) / math.sqrt(32)
    am = s.argmax(-1)
    # with huge margins the output is the value of the arg-max key
    top2 = np.sort(s, -1)[:, -2:]
    sharp = (top2[:, 1] - top2[:, 0]) > 50
    np.testing.assert_allclose(o[0, 0][sharp], v[0, 0][am[sharp]], atol=1e-12)


def test_rows_variant_matches_full():
    q, k, v = (_rand((2, 3, 12, 32), s) for s in (28, 29, 30))
    o = oracle.full_fwd(q, k, v)
    rows = [0, 5, 11, 12, 40, 71]
    np.testing.assert_array_equal(oracle.full_rows(q, k, v, rows), o.reshape(-1, 32)[rows])
