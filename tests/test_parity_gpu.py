"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle on
the same seeded host arrays, element by element.

Every test also checks, through the library's launch counters, that the
kernel family under test really ran (no silent detour).
"""
import math

import numpy as np
import pytest

import oracle
from tests.util import assert_close, errors, to_dev, to_host64
from workloads import WORKLOADS, make_inputs, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ta():
    import torch
    from transformer_attention_tcgen05_gb300.build import build
    build()
    import transformer_attention_tcgen05_gb300 as ta
    torch.cuda.set_device(0)
    return ta


class launched:
    """Context manager asserting that a kernel family launched inside it."""

    def __init__(self, ta, family):
        self.ta, self.family = ta, family

    def __enter__(self):
        self.n0 = self.ta.launch_count(self.family)
        return self

    def __exit__(self, *exc):
        if exc[0] is None:
            assert self.ta.launch_count(self.family) > self.n0, f"{self.family} did not launch"


def _dev(x, w, names="qkv"):
    return [to_dev(x[n], w.dtype) for n in names]


def _f64(x, w, names="qkv"):
    return [to_f64(x[n], w.dtype) for n in names]


# ------------------------------------------------------------ full attention

def test_mha_tiny_fp32(ta):
    w = WORKLOADS["mha_tiny"]
    x = make_inputs(w)
    with launched(ta, "simt"):
        o = ta.full_fwd(*_dev(x, w))
    ref = oracle.full_fwd(*_f64(x, w))
    assert_close(to_host64(o), ref, "f32", "mha_tiny")
    assert ta.device_status() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,Nq,Nkv,D", [
    (1, 1, 1, 1, 32), (2, 3, 17, 33, 32), (1, 2, 130, 257, 64), (1, 2, 200, 129, 128),
    (2, 1, 64, 1000, 128), (1, 1, 257, 255, 64),
])
def test_full_shapes(ta, dtype, B, H, Nq, Nkv, D):
    rng = np.random.Generator(np.random.PCG64(7000 + Nq + Nkv + D))
    from workloads import draw
    q = draw(rng, (B, H, Nq, D), dtype)
    k = draw(rng, (B, H, Nkv, D), dtype)
    v = draw(rng, (B, H, Nkv, D), dtype)
    o = ta.full_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype))
    ref = oracle.full_fwd(to_f64(q, dtype), to_f64(k, dtype), to_f64(v, dtype))
    assert_close(to_host64(o), ref, dtype, f"full {dtype} {B,H,Nq,Nkv,D}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_full_sharp_rows(ta, dtype):
    # Q x 8: peaked rows exercise the running-max rescale
    rng = np.random.Generator(np.random.PCG64(7100))
    from workloads import bf16_round
    q = rng.standard_normal((1, 2, 300, 64), dtype=np.float32) * 8
    k = rng.standard_normal((1, 2, 700, 64), dtype=np.float32)
    v = rng.standard_normal((1, 2, 700, 64), dtype=np.float32)
    if dtype == "bf16":
        q, k, v = bf16_round(q), bf16_round(k), bf16_round(v)
    o = ta.full_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype))
    ref = oracle.full_fwd(to_f64(q, dtype), to_f64(k, dtype), to_f64(v, dtype))
    assert_close(to_host64(o), ref, dtype, f"sharp {dtype}")


def test_explicit_scale_and_determinism(ta):
    import torch
    w = WORKLOADS["mha_tiny"]
    x = make_inputs(w)
    q, k, v = _dev(x, w)
    o1 = ta.full_fwd(q, k, v, scale=0.05)
    o2 = ta.full_fwd(q, k, v, scale=0.05)
    assert torch.equal(o1, o2)
    ref = oracle.full_fwd(*_f64(x, w), scale=0.05)
    assert_close(to_host64(o1), ref, "f32", "scale 0.05")


def test_output_guard_bands_untouched(ta):
    import torch
    w = WORKLOADS["mha_tiny"]
    x = make_inputs(w)
    q, k, v = _dev(x, w)
    n = q.numel()
    buf = torch.full((n + 2048,), 12345.0, device=q.device)
    o = buf[1024:1024 + n].view(q.shape)
    ta.full_fwd(q, k, v, o=o)
    torch.cuda.synchronize()
    assert torch.all(buf[:1024] == 12345.0) and torch.all(buf[1024 + n:] == 12345.0)


# ----------------------------------------------------- neighborhood attention

NA_SMALL = ["na3d_1x4x4_k3x7x7_f32", "na3d_1x4x4_k3x7x7_bf16",
            "na3d_9x64x64_k11_f32", "na3d_9x64x64_k11_bf16"]


@pytest.mark.parametrize("name", NA_SMALL)
def test_na3d_clamp_cases_full_compare(ta, name):
    w = WORKLOADS[name]
    x = make_inputs(w)
    o = ta.na3d_fwd(*_dev(x, w), w.grid, w.kernel)
    ref = oracle.na3d_fwd(*_f64(x, w), w.grid, w.kernel)
    assert_close(to_host64(o), ref, w.dtype, name)
    assert ta.device_status() == 0


def test_na3d_kernel_covering_grid_is_full_attention(ta):
    # the [1,4,4] / k[3,7,7] case: every query attends to all 16 tokens
    w = WORKLOADS["na3d_1x4x4_k3x7x7_f32"]
    x = make_inputs(w)
    q, k, v = _dev(x, w)
    o_na = to_host64(ta.na3d_fwd(q, k, v, w.grid, w.kernel))
    o_full = to_host64(ta.full_fwd(q, k, v))
    np.testing.assert_allclose(o_na, o_full, rtol=0, atol=2e-6)


@pytest.mark.parametrize("grid,kernel", [
    ((1, 4, 4), (3, 7, 7)), ((9, 64, 64), (11, 11, 11)), ((21, 60, 104), (11, 11, 11)),
    ((5, 7, 3), (3, 9, 1)), ((2, 13, 17), (5, 5, 7)),
])
def test_window_starts_bit_exact(ta, grid, kernel):
    with launched(ta, "na_starts"):
        st = ta.na3d_window_starts(grid, kernel).cpu().numpy()
    np.testing.assert_array_equal(st, oracle.na3d_window_starts(grid, kernel))


def test_window_sets_through_the_kernel(ta):
    # black-box probe: Q = 0 makes every output the mean of V over the window;
    # V channels carry (t, h, w, t^2, h^2, w^2, 1): mean and second moment per
    # axis identify each query's interval exactly (small integers, exact fp32)
    import itertools
    grid, kernel = (6, 20, 24), (3, 7, 11)
    T, Hg, W = grid
    N = T * Hg * W
    c = np.array(list(itertools.product(range(T), range(Hg), range(W))), dtype=np.float32)
    v = np.zeros((1, 1, N, 32), dtype=np.float32)
    v[0, 0, :, 0:3] = c
    v[0, 0, :, 3:6] = c ** 2
    v[0, 0, :, 6] = 1
    q = np.zeros_like(v)
    k = np.random.Generator(np.random.PCG64(7200)).standard_normal(v.shape, dtype=np.float32)
    o = to_host64(ta.na3d_fwd(to_dev(q, "f32"), to_dev(k, "f32"), to_dev(v, "f32"), grid, kernel))[0, 0]
    st = oracle.na3d_window_starts(grid, kernel)
    for ax, n in enumerate(grid):
        keff = min(kernel[ax], n)
        lo = st[:, ax].astype(np.float64)
        mean = lo + (keff - 1) / 2
        m2 = np.array([np.mean(np.arange(a, a + keff) ** 2) for a in st[:, ax]])
        np.testing.assert_allclose(o[:, ax], mean, rtol=0, atol=1e-4)
        np.testing.assert_allclose(o[:, 3 + ax], m2, rtol=2e-6, atol=1e-3)


# ------------------------------------------------------------------ decode

def _decode_case(ta, w, check=True):
    import torch
    x = make_inputs(w)
    q, k, v = to_dev(x["q"], "bf16"), to_dev(x["k"], "bf16"), to_dev(x["v"], "bf16")
    sl = torch.from_numpy(x["seq_len"]).cuda()
    with launched(ta, "decode"):
        o = ta.decode_gqa(q, k, v, sl)
    ref = oracle.decode_gqa(to_f64(x["q"], "bf16"), to_f64(x["k"], "bf16"), to_f64(x["v"], "bf16"),
                            x["seq_len"])
    return assert_close(to_host64(o), ref, "bf16", f"decode {w}")


def test_decode_workload_full_size(ta):
    _decode_case(ta, WORKLOADS["gqa_decode"])
    assert ta.device_status() == 0


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 8, 128), (16, 8, 128), (12, 4, 64), (32, 4, 128),
                                      (9, 3, 64), (6, 1, 64)])
def test_decode_groups_and_ragged_lengths(ta, Hq, Hkv, D):
    w = WORKLOADS["gqa_decode"].with_(B=3, H=Hq, Hkv=Hkv, D=D, Lmax=777, seq_len=(1, 777, 300),
                                      seed=7300 + Hq + D)
    _decode_case(ta, w)


def test_decode_workspace_is_reusable_and_deterministic(ta):
    import torch
    w = WORKLOADS["gqa_decode"].with_(B=2, Lmax=1000, seq_len=(1000, 513))
    x = make_inputs(w)
    q, k, v = to_dev(x["q"], "bf16"), to_dev(x["k"], "bf16"), to_dev(x["v"], "bf16")
    sl = torch.from_numpy(x["seq_len"]).cuda()
    ws = torch.zeros(ta.decode_workspace_bytes(2, 32, 8, 1000, 128), dtype=torch.uint8, device="cuda")
    o1 = ta.decode_gqa(q, k, v, sl, workspace=ws)
    o2 = ta.decode_gqa(q, k, v, sl, workspace=ws)
    assert torch.equal(o1, o2)
    ref = oracle.decode_gqa(to_f64(x["q"], "bf16"), to_f64(x["k"], "bf16"), to_f64(x["v"], "bf16"),
                            x["seq_len"])
    assert_close(to_host64(o2), ref, "bf16", "decode reuse")


def test_decode_more_units_than_resident_clusters(ta):
    """1280 (batch, kv-head) units are more than the GPU holds as clusters at
    once, so the splits merge through the workspace (atomic ticket) rather
    than through distributed shared memory; same parity bar."""
    rng = np.random.default_rng(7401)
    sl = tuple(int(x) for x in rng.integers(1, 97, size=160))
    _decode_case(ta, WORKLOADS["gqa_decode"].with_(B=160, H=8, Hkv=8, D=64, Lmax=96, seq_len=sl,
                                                   seed=7401))


def test_decode_rejects_bad_seq_len_on_device(ta):
    import torch
    w = WORKLOADS["gqa_decode"].with_(B=2, Lmax=128)
    x = make_inputs(w)
    q, k, v = to_dev(x["q"], "bf16"), to_dev(x["k"], "bf16"), to_dev(x["v"], "bf16")
    sl = torch.tensor([128, 129], dtype=torch.int32, device="cuda")   # 129 > Lmax
    assert ta.device_status() == 0
    ta.decode_gqa(q, k, v, sl)
    assert ta.device_status() == 6          # ATTN_ERR_DEVICE_CHECK, context still usable
    assert ta.device_status() == 0          # cleared by the read
    _decode_case(ta, w.with_(seq_len=(128, 5)))


# ------------------------------------------------------------ joint + RoPE

def test_joint_small_full_compare(ta):
    import torch
    w = WORKLOADS["flux_joint"].with_(H=3, N=96 + 12 * 20, n_txt=96, img=(12, 20))
    x = make_inputs(w)
    pos = torch.from_numpy(x["pos"]).cuda()
    with launched(ta, "rope"):
        o = ta.rope_joint_fwd(*_dev(x, w), pos)
    ref = oracle.joint_fwd(*_f64(x, w), x["pos"])
    assert_close(to_host64(o), ref, "bf16", "joint small")


def test_joint_fp32_full_compare(ta):
    import torch
    w = WORKLOADS["flux_joint"].with_(dtype="f32", H=2, N=40 + 8 * 9, n_txt=40, img=(8, 9))
    x = make_inputs(w)
    pos = torch.from_numpy(x["pos"]).cuda()
    o = ta.rope_joint_fwd(*_dev(x, w), pos)
    ref = oracle.joint_fwd(*_f64(x, w), x["pos"])
    assert_close(to_host64(o), ref, "f32", "joint fp32")


# ------------------------------------------------- tensor-core (tcgen05) path

@pytest.mark.parametrize("D", [64, 128])
def test_tc_tile_building_blocks(ta, D):
    """The MMA forms on one tile: S = q k^T + q16 k16^T (128B- and 32B-swizzled smem
    operands) and O = P v (TMEM x MN-major smem)."""
    import ctypes
    import torch
    from workloads import bf16_round, bf16_to_f32
    rng = np.random.Generator(np.random.PCG64(7400 + D))
    q = bf16_round(rng.standard_normal((128, D), dtype=np.float32))
    k = bf16_round(rng.standard_normal((128, D), dtype=np.float32))
    v = bf16_round(rng.standard_normal((128, D), dtype=np.float32))
    P = bf16_round(rng.random((128, 128), dtype=np.float32))
    dq, dk, dv, dP = (to_dev(x, "bf16") for x in (q, k, v, P))
    S = torch.empty((128, 128), dtype=torch.float32, device="cuda")
    O = torch.empty((128, D), dtype=torch.float32, device="cuda")
    L = ta.lib()
    L.attn_debug_tc_tile.restype = ctypes.c_int
    st = L.attn_debug_tc_tile(ctypes.c_void_p(dq.data_ptr()), ctypes.c_void_p(dk.data_ptr()),
                              ctypes.c_void_p(dv.data_ptr()), ctypes.c_void_p(dP.data_ptr()),
                              ctypes.c_void_p(S.data_ptr()), ctypes.c_void_p(O.data_ptr()), D,
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    assert ta.device_status() == 0
    f = lambda x: bf16_to_f32(x).astype(np.float64)
    expect_s = f(q) @ f(k).T + f(q)[:, :16] @ f(k)[:, :16].T
    np.testing.assert_allclose(S.cpu().numpy(), expect_s, rtol=0, atol=1e-3)
    np.testing.assert_allclose(O.cpu().numpy(), f(P) @ f(v), rtol=0, atol=1e-3)


@pytest.mark.parametrize("Nq,Nkv,D", [(256, 128, 128), (256, 256, 64), (300, 1000, 128),
                                      (1, 77, 64), (1000, 1, 128), (513, 4100, 64)])
def test_tc_full_parity(ta, Nq, Nkv, D):
    from workloads import draw
    rng = np.random.Generator(np.random.PCG64(7500 + Nq + Nkv + D))
    B, H = 2, 3
    q = draw(rng, (B, H, Nq, D), "bf16")
    k = draw(rng, (B, H, Nkv, D), "bf16")
    v = draw(rng, (B, H, Nkv, D), "bf16")
    with launched(ta, "tc_flash"):
        o = ta.full_fwd(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"))
    ref = oracle.full_fwd(to_f64(q, "bf16"), to_f64(k, "bf16"), to_f64(v, "bf16"))
    assert_close(to_host64(o), ref, "bf16", f"tc full {Nq,Nkv,D}")
    assert ta.device_status() == 0


def test_tc_full_sharp_rows_rescale(ta):
    # Q x 8 and a late key block with large scores: forces the lazy O rescale
    from workloads import bf16_round
    rng = np.random.Generator(np.random.PCG64(7600))
    q = rng.standard_normal((1, 2, 256, 128), dtype=np.float32) * 8
    k = rng.standard_normal((1, 2, 1024, 128), dtype=np.float32)
    k[:, :, 700:720] *= 4
    v = rng.standard_normal((1, 2, 1024, 128), dtype=np.float32)
    q, k, v = bf16_round(q), bf16_round(k), bf16_round(v)
    with launched(ta, "tc_flash"):
        o = ta.full_fwd(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"))
    ref = oracle.full_fwd(to_f64(q, "bf16"), to_f64(k, "bf16"), to_f64(v, "bf16"))
    assert_close(to_host64(o), ref, "bf16", "tc sharp")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("growth", [14.0, 40.0])
@pytest.mark.parametrize("D", [64, 128])
def test_tc_scores_growing_from_tile_to_tile(ta, dtype, growth, D):
    """Each key tile's scores exceed the previous tile's by about `growth` (in
    log2 units).  After the first tile the kernel exponentiates against the
    running maximum as it stands: a growth of 40 overflows the tile's row sum
    every time (the tile is redone with its own maximum and O rescaled); a
    growth of 14 keeps P up to ~2^14 in bf16 but passes f16's bound (redo)."""
    from workloads import bf16_round
    rng = np.random.Generator(np.random.PCG64(7700 + D + int(growth)))
    H, Nq, Nkv = 2, 256, 5 * 128
    u = np.where(rng.random(D) < 0.5, -1.0, 1.0).astype(np.float32)
    alpha = np.repeat(np.arange(5, dtype=np.float32), 128) * growth / (1.4426950408889634 * math.sqrt(D))
    q = u + 0.25 * rng.standard_normal((1, H, Nq, D), dtype=np.float32)
    k = alpha[None, None, :, None] * u + 0.5 * rng.standard_normal((1, H, Nkv, D), dtype=np.float32)
    v = rng.standard_normal((1, H, Nkv, D), dtype=np.float32)
    rnd = bf16_round if dtype == "bf16" else (lambda a: a.astype(np.float16))
    q, k, v = rnd(q), rnd(k), rnd(v)
    with launched(ta, "tc_flash"):
        o = ta.full_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype))
    ref = oracle.full_fwd(to_f64(q, dtype), to_f64(k, dtype), to_f64(v, dtype))
    assert_close(to_host64(o), ref, dtype, f"growing scores {dtype} D={D} growth={growth}")
    assert ta.device_status() == 0


def test_flux_joint_full_size_sampled_rows(ta):
    import torch
    w = WORKLOADS["flux_joint"]
    x = make_inputs(w)
    pos = torch.from_numpy(x["pos"]).cuda()
    with launched(ta, "tc_flash"), launched(ta, "rope"):
        o = ta.rope_joint_fwd(*_dev(x, w), pos)
    rng = np.random.default_rng(11)
    N = w.N
    rows = np.concatenate([rng.choice(w.B * w.H * N, 2048, replace=False),
                           [0, N - 1, 511, 512, 513, N * w.H - 1]])
    rows = np.unique(rows)
    ref = oracle.joint_fwd(*_f64(x, w), x["pos"], rows=rows)
    got = to_host64(o).reshape(-1, w.D)[rows]
    assert_close(got, ref, "bf16", "flux joint sampled")
    assert ta.device_status() == 0


@pytest.mark.parametrize("grid,kernel,H", [((6, 20, 24), (3, 7, 11), 2), ((9, 16, 16), (11, 11, 11), 1),
                                           ((3, 9, 40), (5, 3, 9), 2), ((1, 4, 4), (3, 7, 7), 2),
                                           ((13, 17, 19), (7, 9, 5), 1),
                                           # several (box, head) items per stream
                                           ((3, 9, 40), (5, 3, 9), 48), ((6, 20, 24), (3, 7, 11), 24)])
def test_tc_na3d_parity(ta, grid, kernel, H):
    w = WORKLOADS["na3d_21x60x104_k11"].with_(grid=grid, kernel=kernel, H=H,
                                             N=int(np.prod(grid)), seed=7700 + sum(grid))
    x = make_inputs(w)
    with launched(ta, "tc_na"):
        o = ta.na3d_fwd(*_dev(x, w), w.grid, w.kernel)
    ref = oracle.na3d_fwd(*_f64(x, w), w.grid, w.kernel)
    assert_close(to_host64(o), ref, "bf16", f"tc na3d {grid} {kernel}")
    assert ta.device_status() == 0


def test_tc_na3d_batch_parity(ta):
    """Batch and heads together index the kernel's (box, head) items:
    B = 3 batches of 5 heads, several items per stream."""
    w = WORKLOADS["na3d_21x60x104_k11"].with_(B=3, H=5, grid=(3, 9, 40), kernel=(5, 3, 9),
                                             N=3 * 9 * 40, seed=7790)
    x = make_inputs(w)
    with launched(ta, "tc_na"):
        o = ta.na3d_fwd(*_dev(x, w), w.grid, w.kernel)
    ref = oracle.na3d_fwd(*_f64(x, w), w.grid, w.kernel)
    assert ref.shape[0] == 3
    assert_close(to_host64(o), ref, "bf16", "tc na3d batch 3")
    assert ta.device_status() == 0


def test_na3d_large_full_size_sampled_rows(ta):
    w = WORKLOADS["na3d_21x60x104_k11"]
    x = make_inputs(w)
    with launched(ta, "tc_na"):
        o = ta.na3d_fwd(*_dev(x, w), w.grid, w.kernel)
    T, Hg, W = w.grid
    rng = np.random.default_rng(12)
    N = w.N
    # a seeded sample plus rows on every face, edge and corner of the grid
    picks = [(t, h, ww) for t in (0, 1, 5, 10, 15, 19, 20) for h in (0, 4, 5, 30, 54, 55, 59)
             for ww in (0, 3, 5, 50, 98, 100, 103)]
    edge = np.array([(t * Hg + h) * W + ww for t, h, ww in picks])
    rows = np.unique(np.concatenate([rng.choice(w.B * w.H * N, 3000, replace=False),
                                     edge, edge + 3 * N, edge + 7 * N]))
    ref = oracle.na3d_fwd(*_f64(x, w), w.grid, w.kernel, rows=rows)
    got = to_host64(o).reshape(-1, w.D)[rows]
    assert_close(got, ref, "bf16", "na3d large sampled")
    assert ta.device_status() == 0


@pytest.mark.parametrize("scale", [0.01, 1.0])
def test_tc_na3d_explicit_scale(ta, scale):
    # the window penalty channels are sized from the scale: tiny and large scales
    w = WORKLOADS["na3d_21x60x104_k11"].with_(grid=(5, 12, 20), kernel=(3, 5, 7), H=1, N=5 * 12 * 20,
                                             seed=7800 + int(scale * 100))
    x = make_inputs(w)
    with launched(ta, "tc_na"):
        o = ta.na3d_fwd(*_dev(x, w), w.grid, w.kernel, scale=scale)
    ref = oracle.na3d_fwd(*_f64(x, w), w.grid, w.kernel, scale=scale)
    assert_close(to_host64(o), ref, "bf16", f"tc na3d scale {scale}")


# ------------------------------------------- graph-stable decode step (append)

def test_kv_append_writes_at_device_position_and_advances(ta):
    import torch
    from workloads import draw
    B, Hkv, Lmax, D = 3, 2, 40, 64
    rng = np.random.Generator(np.random.PCG64(8100))
    kc = to_dev(draw(rng, (B, Hkv, Lmax, D), "bf16"), "bf16")
    vc = to_dev(draw(rng, (B, Hkv, Lmax, D), "bf16"), "bf16")
    kn = to_dev(draw(rng, (B, Hkv, D), "bf16"), "bf16")
    vn = to_dev(draw(rng, (B, Hkv, D), "bf16"), "bf16")
    k0, v0 = kc.clone(), vc.clone()
    sl = torch.tensor([0, 17, 39], dtype=torch.int32, device="cuda")
    with launched(ta, "kv_append"):
        ta.kv_append(kc, vc, kn, vn, sl)
    assert sl.tolist() == [1, 18, 40]
    for b, pos in enumerate([0, 17, 39]):
        assert torch.equal(kc[b, :, pos], kn[b]) and torch.equal(vc[b, :, pos], vn[b])
        k0[b, :, pos] = kn[b]
        v0[b, :, pos] = vn[b]
    assert torch.equal(kc, k0) and torch.equal(vc, v0)          # nothing else touched
    # a full cache (position == Lmax) is refused on the device and left untouched
    assert ta.device_status() == 0
    ta.kv_append(kc, vc, kn, vn, torch.tensor([1, 18, 40], dtype=torch.int32, device="cuda"))
    assert ta.device_status() == 6


def test_decode_step_captured_once_and_replayed_per_token(ta):
    """Append + decode captured in one CUDA graph, replayed for several tokens
    with unchanged arguments (positions live on the device)."""
    import torch
    from workloads import draw
    w = WORKLOADS["gqa_decode"].with_(B=2, Lmax=300, seq_len=(100, 257), seed=8200)
    x = make_inputs(w)
    rng = np.random.Generator(np.random.PCG64(8201))
    kc, vc = to_dev(x["k"], "bf16"), to_dev(x["v"], "bf16")
    kc_host, vc_host = to_f64(x["k"], "bf16"), to_f64(x["v"], "bf16")
    lens = list(x["seq_len"])
    sl = torch.from_numpy(x["seq_len"]).cuda()
    B, Hq, Hkv, D = w.B, w.H, w.Hkv, w.D
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros((B, Hkv, D), dtype=torch.bfloat16, device="cuda")
    vn = torch.zeros_like(kn)
    o = torch.empty_like(q)
    ws = torch.zeros(ta.decode_workspace_bytes(B, Hq, Hkv, w.Lmax, D), dtype=torch.uint8,
                     device="cuda")
    # first calls outside the capture (per-device set-up of the library)
    sl_warm = sl.clone()
    kc_w, vc_w = kc.clone(), vc.clone()
    ta.kv_append(kc_w, vc_w, kn, vn, sl_warm)
    ta.decode_gqa(q, kc_w, vc_w, sl_warm, o=o, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ta.kv_append(kc, vc, kn, vn, sl)
        ta.decode_gqa(q, kc, vc, sl, o=o, workspace=ws)
    for step in range(3):
        qh, knh, vnh = (draw(rng, shp, "bf16") for shp in ((B, Hq, D), (B, Hkv, D), (B, Hkv, D)))
        q.copy_(to_dev(qh, "bf16"))
        kn.copy_(to_dev(knh, "bf16"))
        vn.copy_(to_dev(vnh, "bf16"))
        g.replay()
        torch.cuda.synchronize()
        for b in range(B):
            kc_host[b, :, lens[b]] = to_f64(knh, "bf16")[b]
            vc_host[b, :, lens[b]] = to_f64(vnh, "bf16")[b]
            lens[b] += 1
        assert sl.tolist() == lens
        ref = oracle.decode_gqa(to_f64(qh, "bf16"), kc_host, vc_host, np.array(lens, np.int32))
        assert_close(to_host64(o), ref, "bf16", f"graph decode step {step}")
    assert ta.device_status() == 0


# ------------------------------------------------------ causal GQA prefill

@pytest.mark.parametrize("dtype,B,Hq,Hkv,N,D", [
    ("bf16", 1, 4, 1, 256, 128), ("bf16", 2, 8, 2, 300, 64), ("bf16", 1, 2, 2, 1000, 128),
    ("bf16", 1, 6, 3, 1, 64), ("bf16", 1, 4, 2, 129, 32), ("f32", 2, 4, 2, 200, 64),
    ("f32", 1, 3, 1, 70, 32),
])
def test_causal_gqa_parity(ta, dtype, B, Hq, Hkv, N, D):
    from workloads import draw
    rng = np.random.Generator(np.random.PCG64(8300 + N + D + Hq))
    q = draw(rng, (B, Hq, N, D), dtype)
    k = draw(rng, (B, Hkv, N, D), dtype)
    v = draw(rng, (B, Hkv, N, D), dtype)
    family = "tc_flash" if (dtype == "bf16" and D >= 64) else "simt"
    with launched(ta, family):
        o = ta.causal_gqa_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype))
    ref = oracle.causal_gqa_fwd(to_f64(q, dtype), to_f64(k, dtype), to_f64(v, dtype))
    assert_close(to_host64(o), ref, dtype, f"causal gqa {dtype} {B,Hq,Hkv,N,D}")
    assert ta.device_status() == 0


def test_causal_gqa_llama_prefill_sampled_rows(ta):
    # a Llama-8B-like grouped prefill: 32 query heads on 8 KV heads, 4096 tokens
    from workloads import draw
    B, Hq, Hkv, N, D = 1, 32, 8, 4096, 128
    rng = np.random.Generator(np.random.PCG64(8400))
    q, k, v = (draw(rng, s, "bf16") for s in ((B, Hq, N, D), (B, Hkv, N, D), (B, Hkv, N, D)))
    o = ta.causal_gqa_fwd(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"))
    rows = np.unique(np.concatenate([np.random.default_rng(13).choice(B * Hq * N, 1500, replace=False),
                                     [0, 1, 127, 128, 255, 256, N - 1, 31 * N + N - 1]]))
    ref = oracle.causal_gqa_fwd(to_f64(q, "bf16"), to_f64(k, "bf16"), to_f64(v, "bf16"), rows=rows)
    assert_close(to_host64(o).reshape(-1, D)[rows], ref, "bf16", "llama prefill sampled")
