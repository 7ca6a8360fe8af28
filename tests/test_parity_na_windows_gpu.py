"""Window index sets through the tensor-core neighborhood kernel, bit-exact.

The NATTEN boundary rule of candle PR #11 ("kernel exceeds grid extent"
commit): per axis k_eff = min(k, n), window [s, s + k_eff) with
s = clamp(i - k/2, 0, n - k_eff); the 3D window is the Cartesian product.

These tests send 16-bit (bf16 and f16) inputs with D = 64 through
attn_na3d_fwd, so the tcgen05 neighborhood kernel runs (asserted by its launch
counter), and read every query's window set back out of the output:

  * Q = 0 makes every admitted score exactly 0, so every admitted key gets
    P = 1 and every masked key P = 0, whatever the mask mechanism;
  * V channel 0..2 hold the key's (t, h, w) and channel 3 holds 1: the output
    is the mean coordinate over the window, s + (k_eff - 1) / 2 per axis,
    a half-integer below 128, exact in both 16-bit types;
  * V channels 4..63 hold a one-hot code of one axis' coordinate (60 values
    per call, several calls per grid): output channel 4 + j is
    count(window keys with that coordinate) / |window|, i.e. 1 / k_eff for a
    coordinate inside the axis interval and exactly 0 outside it.  Any extra
    or missing key changes a count and so the rounded value (counts are at
    most 128 here, so a count that is off by one moves the quotient by more
    than one unit in the last place).

The expected arrays come from the oracle's window starts (pinned on the CPU
against a brute-force search of the window); the comparison is exact equality
on every row, head and channel.

A second test plants, for queries just outside its window, one key whose raw
score exceeds every in-window score by far more than any fixed penalty that
depends on the scale alone: the masked key must still get P = 0.
"""
import itertools

import numpy as np
import pytest

import oracle
from tests.util import assert_close, to_dev, to_host64
from workloads import bf16_round, bf16_to_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ta():
    import torch
    from transformer_attention_tcgen05_gb300.build import build
    build()
    import transformer_attention_tcgen05_gb300 as ta
    torch.cuda.set_device(0)
    return ta


def _round(x: np.ndarray, dtype: str) -> np.ndarray:
    """float64 -> the 16-bit storage type (round to nearest even), widened back."""
    x32 = np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_to_f32(bf16_round(x32)).astype(np.float64)
    return x32.astype(np.float16).astype(np.float64)


def _storage(x: np.ndarray, dtype: str) -> np.ndarray:
    x32 = np.asarray(x, dtype=np.float32)
    return bf16_round(x32) if dtype == "bf16" else x32.astype(np.float16)


def _dev(x: np.ndarray, dtype: str):
    import torch
    if dtype == "bf16":
        return to_dev(x, "bf16")
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


# (grid, kernel, heads): the pages' two clamp shapes at D = 64, the large
# workload's grid, and odd/even extents where windows clamp on some axes.  The
# kernel runs one CTA per SM with two streams of (box, head) items, so the
# many-head cases give every stream several boxes whose window geometry
# changes from one to the next; (1, 4, 4) is one box per head, so one head
# leaves the second stream without work and seven give the last CTA one box.
CASES = [
    ((9, 64, 64), (11, 11, 11), 1),
    ((21, 60, 104), (11, 11, 11), 1),
    ((1, 4, 4), (3, 7, 7), 2),
    ((1, 4, 4), (3, 7, 7), 1),
    ((1, 4, 4), (3, 7, 7), 7),
    ((4, 6, 33), (5, 7, 9), 1),
    ((2, 5, 16), (3, 5, 17), 1),
    ((7, 8, 9), (7, 9, 11), 2),
    ((3, 11, 50), (1, 3, 49), 1),
    ((5, 1, 30), (9, 5, 3), 1),
    ((1, 4, 4), (3, 7, 7), 400),
    ((4, 6, 33), (5, 7, 9), 64),
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("grid,kernel,H", CASES)
def test_window_sets_bit_exact_through_the_tensor_core_kernel(ta, dtype, grid, kernel, H):
    import torch
    T, Hg, W = grid
    N, D = T * Hg * W, 64
    coords = np.array(list(itertools.product(range(T), range(Hg), range(W))), dtype=np.int64)
    starts = oracle.na3d_window_starts(grid, kernel).astype(np.int64)     # [N, 3]
    keff = [min(kk, n) for kk, n in zip(kernel, grid)]
    q = torch.zeros((1, H, N, D), dtype=torch.bfloat16 if dtype == "bf16" else torch.float16,
                    device="cuda")
    k = _dev(_storage(np.random.default_rng(8800).standard_normal((1, H, N, D)), dtype), dtype)

    mean = np.stack([starts[:, a] + (keff[a] - 1) / 2 for a in range(3)], axis=1)
    runs = [(a, c0) for a in range(3) for c0 in range(0, grid[a], 60)]
    for a, c0 in runs:
        v = np.zeros((N, D), dtype=np.float64)
        v[:, 0:3] = coords
        v[:, 3] = 1.0
        width = min(60, grid[a] - c0)
        for j in range(width):
            v[:, 4 + j] = coords[:, a] == c0 + j
        vd = _dev(np.broadcast_to(_storage(v, dtype), (1, H, N, D)).copy(), dtype)
        n0 = ta.launch_count("tc_na")
        o = ta.na3d_fwd(q, k, vd, grid, kernel)
        assert ta.launch_count("tc_na") > n0, "the tensor-core neighborhood kernel did not run"
        got = to_host64(o)
        # expected: per-axis window means, ones, and the one-hot membership
        exp = np.zeros((N, D), dtype=np.float64)
        exp[:, 0:3] = mean
        exp[:, 3] = 1.0
        cj = c0 + np.arange(width)
        inside = (cj[None, :] >= starts[:, a:a + 1]) & (cj[None, :] < starts[:, a:a + 1] + keff[a])
        exp[:, 4:4 + width] = np.where(inside, 1.0 / keff[a], 0.0)
        exp = _round(exp, dtype)
        for h in range(H):
            bad = np.nonzero(np.any(got[0, h] != exp, axis=1))[0]
            assert bad.size == 0, (
                f"{dtype} {grid}/{kernel} axis {a} from {c0}, head {h}: {bad.size} rows with a "
                f"wrong window; first row {bad[0]} at {tuple(coords[bad[0]])}: got "
                f"{got[0, h, bad[0], :8]} / {got[0, h, bad[0], 4:4 + width].nonzero()[0] + c0}, "
                f"expected {exp[bad[0], :8]} / starts {starts[bad[0]]}")
    assert ta.device_status() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_masked_key_with_a_far_higher_score_stays_masked(ta, dtype):
    """Keys equal to 60 u score about 692 (in log2 units) against queries near
    u, far above every in-window score (about 0).  For the queries whose window
    just misses such a key it must contribute exactly nothing."""
    grid, kernel, H, D = (6, 20, 24), (3, 7, 11), 1, 64
    T, Hg, W = grid
    N = T * Hg * W
    g = np.random.default_rng(8900)
    u = np.where(g.random(D) < 0.5, -1.0, 1.0)
    q = u + 0.1 * g.standard_normal((1, H, N, D))
    k = 0.5 * g.standard_normal((1, H, N, D))
    v = g.standard_normal((1, H, N, D))
    poison = g.choice(N, 24, replace=False)
    k[:, :, poison] = 60.0 * u
    q, k, v = (_storage(x, dtype) for x in (q, k, v))
    n0 = ta.launch_count("tc_na")
    o = ta.na3d_fwd(_dev(q, dtype), _dev(k, dtype), _dev(v, dtype), grid, kernel)
    assert ta.launch_count("tc_na") > n0, "the tensor-core neighborhood kernel did not run"
    wide = (lambda x: bf16_to_f32(x).astype(np.float64)) if dtype == "bf16" else \
        (lambda x: x.astype(np.float64))
    ref = oracle.na3d_fwd(wide(q), wide(k), wide(v), grid, kernel)
    assert_close(to_host64(o), ref, dtype, f"{dtype} masked high-score keys")
    assert ta.device_status() == 0
