"""Independent brute-force attention in numpy, used only to pin the oracle.

It is deliberately built differently from the oracle:
  * the whole dense N x N score matrix is formed at once;
  * the neighborhood window is found by search -- among all length-k_eff
    intervals inside [0, n) that contain i, the one whose centre is nearest to
    i -- instead of the clamp formula;
  * softmax is taken without max subtraction (tiny magnitudes only).
"""
from __future__ import annotations

import itertools

import numpy as np


def window_by_search(i: int, n: int, k: int) -> range:
    """Window of position i on an axis of extent n for a requested odd kernel k."""
    keff = min(k, n)
    best = None
    for s in range(0, n - keff + 1):
        if not (s <= i < s + keff):
            continue
        centre2 = 2 * s + keff - 1          # twice the centre (exact for any parity)
        dist = abs(centre2 - 2 * i)
        if best is None or dist < best[0]:
            best = (dist, s)
    assert best is not None
    return range(best[1], best[1] + keff)


def na3d_mask(grid, kernel) -> np.ndarray:
    """Boolean [N, N] mask, True where key j is in query i's 3D window."""
    T, Hg, W = grid
    N = T * Hg * W
    m = np.zeros((N, N), dtype=bool)
    coords = list(itertools.product(range(T), range(Hg), range(W)))
    for i, (t, h, w) in enumerate(coords):
        wt = window_by_search(t, T, kernel[0])
        wh = window_by_search(h, Hg, kernel[1])
        ww = window_by_search(w, W, kernel[2])
        for a in wt:
            for b in wh:
                for c in ww:
                    m[i, (a * Hg + b) * W + c] = True
    return m


def dense_attention(q, k, v, scale, mask=None):
    """q [..., Nq, D], k/v [..., Nkv, D]; mask [Nq, Nkv] bool or None."""
    s = np.einsum("...id,...jd->...ij", q, k) * scale
    e = np.exp(s)
    if mask is not None:
        e = np.where(mask, e, 0.0)
    p = e / e.sum(axis=-1, keepdims=True)
    return np.einsum("...ij,...jd->...id", p, v), p
