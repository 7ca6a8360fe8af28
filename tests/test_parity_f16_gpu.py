"""GPU parity for the F16 dtype (IEEE half storage, candle's third `Map3`
type) on every entry point, against the same fp64 oracle as bf16 and fp32.

The inputs are the float32 N(0,1) draws rounded to f16; the oracle widens them
exactly, so only the kernels' own rounding (P and O to f16) and fp32
accumulation are measured, against the f16 bounds in tests/util.py.
"""
import numpy as np
import pytest

import oracle
from tests.util import assert_close, to_dev, to_host64
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


def _ran(ta, family, n0):
    assert ta.launch_count(family) > n0, f"{family} did not launch"


def _io(w, names="qkv"):
    x = make_inputs(w)
    return x, [to_dev(x[n], "f16") for n in names], [to_f64(x[n], "f16") for n in names]


@pytest.mark.parametrize("H,Nq,Nkv,D,family", [(2, 300, 333, 128, "tc_flash"),
                                                (3, 257, 200, 64, "tc_flash"),
                                                (2, 70, 90, 32, "simt")])
def test_f16_full(ta, H, Nq, Nkv, D, family):
    import torch
    g = np.random.default_rng(9100 + D)
    q = g.standard_normal((1, H, Nq, D), dtype=np.float32).astype(np.float16)
    k = g.standard_normal((1, H, Nkv, D), dtype=np.float32).astype(np.float16)
    v = g.standard_normal((1, H, Nkv, D), dtype=np.float32).astype(np.float16)
    n0 = ta.launch_count(family)
    o = ta.full_fwd(*(torch.from_numpy(a).cuda() for a in (q, k, v)))
    _ran(ta, family, n0)
    assert o.dtype == torch.float16
    ref = oracle.full_fwd(*(a.astype(np.float64) for a in (q, k, v)))
    assert_close(to_host64(o), ref, "f16", f"f16 full {H, Nq, Nkv, D}")
    assert ta.device_status() == 0


def test_f16_joint_rope(ta):
    import torch
    w = WORKLOADS["flux_joint"].with_(dtype="f16", H=3, N=96 + 12 * 20, n_txt=96, img=(12, 20),
                                      seed=9200)
    x, dev, f64 = _io(w)
    n0 = ta.launch_count("rope")
    o = ta.rope_joint_fwd(*dev, torch.from_numpy(x["pos"]).cuda())
    _ran(ta, "rope", n0)
    ref = oracle.joint_fwd(*f64, x["pos"])
    assert_close(to_host64(o), ref, "f16", "f16 joint")


@pytest.mark.parametrize("Hq,Hkv,N,D", [(4, 2, 300, 128), (6, 3, 257, 64)])
def test_f16_causal_gqa(ta, Hq, Hkv, N, D):
    import torch
    g = np.random.default_rng(9300 + D)
    q = g.standard_normal((1, Hq, N, D), dtype=np.float32).astype(np.float16)
    k = g.standard_normal((1, Hkv, N, D), dtype=np.float32).astype(np.float16)
    v = g.standard_normal((1, Hkv, N, D), dtype=np.float32).astype(np.float16)
    n0 = ta.launch_count("tc_flash")
    o = ta.causal_gqa_fwd(*(torch.from_numpy(a).cuda() for a in (q, k, v)))
    _ran(ta, "tc_flash", n0)
    ref = oracle.causal_gqa_fwd(*(a.astype(np.float64) for a in (q, k, v)))
    assert_close(to_host64(o), ref, "f16", f"f16 causal {Hq, Hkv, N, D}")


@pytest.mark.parametrize("grid,kernel,D,family", [((3, 20, 24), (3, 5, 7), 64, "tc_na"),
                                                  ((5, 9, 33), (11, 11, 11), 64, "tc_na"),
                                                  ((1, 4, 4), (3, 7, 7), 32, "simt")])
def test_f16_na3d(ta, grid, kernel, D, family):
    w = WORKLOADS["na3d_9x64x64_k11_bf16"].with_(dtype="f16", grid=grid, kernel=kernel, D=D, H=2,
                                                 N=grid[0] * grid[1] * grid[2], seed=9400 + D)
    x, dev, f64 = _io(w)
    n0 = ta.launch_count(family)
    o = ta.na3d_fwd(*dev, grid, kernel)
    _ran(ta, family, n0)
    ref = oracle.na3d_fwd(*f64, grid, kernel)
    assert_close(to_host64(o), ref, "f16", f"f16 na3d {grid} {kernel}")
    assert ta.device_status() == 0


def test_f16_na3d_small_scale(ta):
    """A tiny scale: the f16 neighborhood kernel tests h and w per key in the
    softmax (no penalty that f16 would have to hold), so it stays on the
    tensor cores and must still be right."""
    grid, kernel = (3, 20, 24), (3, 5, 7)
    w = WORKLOADS["na3d_9x64x64_k11_bf16"].with_(dtype="f16", grid=grid, kernel=kernel, D=64, H=1,
                                                 N=grid[0] * grid[1] * grid[2], seed=9450)
    x, dev, f64 = _io(w)
    n0 = ta.launch_count("tc_na")
    o = ta.na3d_fwd(*dev, grid, kernel, scale=1e-4)
    _ran(ta, "tc_na", n0)
    ref = oracle.na3d_fwd(*f64, grid, kernel, scale=1e-4)
    assert_close(to_host64(o), ref, "f16", "f16 na3d tiny scale")


@pytest.mark.parametrize("Hq,Hkv,D", [(16, 4, 128), (8, 8, 64)])
def test_f16_decode(ta, Hq, Hkv, D):
    import torch
    w = WORKLOADS["gqa_decode"].with_(dtype="f16", B=3, H=Hq, Hkv=Hkv, D=D, Lmax=777,
                                      seq_len=(1, 777, 300), seed=9500 + Hq + D)
    x, dev, f64 = _io(w)
    n0 = ta.launch_count("decode")
    o = ta.decode_gqa(*dev, torch.from_numpy(x["seq_len"]).cuda())
    _ran(ta, "decode", n0)
    ref = oracle.decode_gqa(*f64, x["seq_len"])
    assert_close(to_host64(o), ref, "f16", f"f16 decode {Hq, Hkv, D}")


def test_f16_kv_append_then_decode(ta):
    import torch
    B, Hq, Hkv, L, D = 2, 8, 2, 64, 128
    g = np.random.default_rng(9600)
    kc = g.standard_normal((B, Hkv, L, D), dtype=np.float32).astype(np.float16)
    vc = g.standard_normal((B, Hkv, L, D), dtype=np.float32).astype(np.float16)
    kn = g.standard_normal((B, Hkv, D), dtype=np.float32).astype(np.float16)
    vn = g.standard_normal((B, Hkv, D), dtype=np.float32).astype(np.float16)
    q = g.standard_normal((B, Hq, D), dtype=np.float32).astype(np.float16)
    sl = np.array([10, 63], dtype=np.int32)
    dkc, dvc = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    dsl = torch.from_numpy(sl).cuda()
    ta.kv_append(dkc, dvc, torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(), dsl)
    assert dsl.cpu().tolist() == [11, 64]
    kc2, vc2 = kc.copy(), vc.copy()
    for b in range(B):
        kc2[b, :, sl[b]] = kn[b]
        vc2[b, :, sl[b]] = vn[b]
    assert np.array_equal(dkc.cpu().numpy(), kc2) and np.array_equal(dvc.cpu().numpy(), vc2)
    o = ta.decode_gqa(torch.from_numpy(q).cuda(), dkc, dvc, dsl)
    ref = oracle.decode_gqa(q.astype(np.float64), kc2.astype(np.float64), vc2.astype(np.float64),
                            sl + 1)
    assert_close(to_host64(o), ref, "f16", "f16 append + decode")
