"""Pins for the oracle's 3D neighborhood attention and its window rule.

Sources: candle PR #11 (commit "kernel exceeds grid extent": effective_kernel()
clamps each axis to min(kernel, extent); a window wider than its axis becomes
full attention on that axis; validate() only requires a positive odd kernel;
repro shapes [9,64,64]/k[11,11,11] and [1,4,4]/k[3,7,7]).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests.brute import dense_attention, na3d_mask, window_by_search

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_window_start_exhaustive_vs_search():
    for n in range(1, 13):
        for k in range(1, 14, 2):
            for i in range(n):
                st = oracle.na_window_start(i, n, k)
                w = window_by_search(i, n, k)
                assert st == w.start, (i, n, k)


def test_window_properties():
    for n in range(1, 30):
        for k in range(1, 22, 2):
            keff = min(k, n)
            for i in range(n):
                st = oracle.na_window_start(i, n, k)
                assert 0 <= st and st + keff <= n           # in bounds
                assert st <= i < st + keff                   # contains the query
                if k // 2 <= i <= n - 1 - k // 2 and k <= n:
                    assert st == i - k // 2                  # centred away from borders


def test_golden_clamp_cases():
    g = json.load(open(os.path.join(GOLD, "na_clamp_cases.json")))
    small, big = g["cases"]
    st = oracle.na3d_window_starts(small["grid"], small["kernel"])
    assert np.all(st == 0)          # every axis clamps to the full extent
    st = oracle.na3d_window_starts(big["grid"], big["kernel"])
    assert np.all(st[:, 0] == big["t_window_all_queries"][0])
    for i, s in big["hw_starts"].items():
        assert oracle.na_window_start(int(i), 64, 11) == s
    T, Hg, W = big["grid"]
    # h-start of token (t, h, w) depends only on h; w-start only on w
    idx = np.arange(T * Hg * W)
    h, w = (idx // W) % Hg, idx % W
    exp_h = np.clip(h - 5, 0, 53)
    exp_w = np.clip(w - 5, 0, 53)
    np.testing.assert_array_equal(st[:, 1], exp_h)
    np.testing.assert_array_equal(st[:, 2], exp_w)


@pytest.mark.parametrize("grid,kernel", [
    ((1, 4, 4), (3, 7, 7)),      # every axis clamps, two even extents
    ((3, 5, 6), (3, 3, 5)),
    ((2, 6, 7), (5, 3, 3)),      # t clamps to 2
    ((4, 4, 5), (1, 1, 3)),
    ((5, 3, 8), (3, 5, 7)),
])
def test_na3d_vs_bruteforce_and_sdpa(grid, kernel):
    B, H, D = 2, 2, 8
    N = int(np.prod(grid))
    q, k, v = (_rand((B, H, N, D), s) for s in (31, 32, 33))
    o, p = oracle.na3d_fwd(q, k, v, grid, kernel, return_p=True)
    mask = na3d_mask(grid, kernel)
    ref, pref = dense_attention(q, k, v, 1 / math.sqrt(D), mask)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(p, pref, rtol=0, atol=1e-13)
    # the admitted set is exactly the mask
    np.testing.assert_array_equal(p[0, 0] > 0, mask)
    keff = [min(a, b) for a, b in zip(kernel, grid)]
    assert np.all(mask.sum(-1) == np.prod(keff))
    t = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=torch.from_numpy(mask)).numpy()
    np.testing.assert_allclose(o, t, rtol=0, atol=1e-12)


def test_kernel_covering_grid_equals_full_attention():
    grid, D = (3, 4, 5), 16
    N = 60
    q, k, v = (_rand((1, 3, N, D), s) for s in (34, 35, 36))
    for kern in [(3, 5, 5), (5, 7, 9), (11, 11, 11)]:
        o = oracle.na3d_fwd(q, k, v, grid, kern)
        np.testing.assert_allclose(o, oracle.full_fwd(q, k, v), rtol=0, atol=1e-13)


def test_zero_q_gives_window_mean_identifying_the_window():
    grid, kernel = (4, 9, 10), (3, 5, 7)
    T, Hg, W = grid
    N = T * Hg * W
    coords = np.array(list(itertools.product(range(T), range(Hg), range(W))), dtype=np.float64)
    v = np.zeros((1, 1, N, 8))
    v[0, 0, :, 0:3] = coords
    v[0, 0, :, 3:6] = coords ** 2
    v[0, 0, :, 6] = 1.0
    q = np.zeros((1, 1, N, 8))
    k = _rand((1, 1, N, 8), 37)
    o = oracle.na3d_fwd(q, k, v, grid, kernel)[0, 0]
    for i, (t, h, w) in enumerate(coords.astype(int)):
        for ax, (c, n, kk) in enumerate(zip((t, h, w), grid, kernel)):
            win = window_by_search(c, n, kk)
            assert abs(o[i, ax] - np.mean(list(win))) < 1e-12
            assert abs(o[i, 3 + ax] - np.mean(np.array(list(win)) ** 2)) < 1e-10
        assert abs(o[i, 6] - 1.0) < 1e-14


def test_page_repro_shape_rows_match_bruteforce():
    # [9,64,64] / k11, sampled rows including borders, vs a brute-force row
    grid, kernel, D = (9, 64, 64), (11, 11, 11), 32
    N = 9 * 64 * 64
    q, k, v = (_rand((1, 1, N, D), s) for s in (38, 39, 40))
    T, Hg, W = grid
    picks = [(0, 0, 0), (8, 63, 63), (4, 5, 6), (2, 58, 0), (6, 31, 63), (1, 53, 10)]
    rows = [(t * Hg + h) * W + w for t, h, w in picks]
    o = oracle.na3d_fwd(q, k, v, grid, kernel, rows=rows)
    for r, (t, h, w) in enumerate(picks):
        keys = [(a * Hg + b) * W + c for a in window_by_search(t, T, 11)
                for b in window_by_search(h, Hg, 11) for c in window_by_search(w, W, 11)]
        assert len(keys) == 1089
        ref, _ = dense_attention(q[0, 0, rows[r]][None], k[0, 0, keys], v[0, 0, keys],
                                 1 / math.sqrt(D))
        np.testing.assert_allclose(o[r], ref[0], rtol=0, atol=1e-12)


def test_rows_variant_matches_full():
    grid, kernel = (3, 6, 7), (3, 5, 3)
    q, k, v = (_rand((2, 2, 126, 16), s) for s in (41, 42, 43))
    o = oracle.na3d_fwd(q, k, v, grid, kernel)
    rows = [0, 1, 125, 126, 300, 503]
    np.testing.assert_array_equal(oracle.na3d_fwd(q, k, v, grid, kernel, rows=rows),
                                  o.reshape(-1, 16)[rows])
