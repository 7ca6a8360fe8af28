"""GPU parity for attention on strided views (attn_full_fwd_strided).

The views are those a model hands over without a copy: the [B, N, H, D]
projection layout read as [B, H, N, D], the three slices of one packed QKV
tensor, and an output written into a column block of a wider buffer.  Each
case is checked against the fp64 oracle on the values the views hold, and
against the contiguous entry point on the same values: the two calls run the
same kernel with the same arithmetic order, so they agree bit for bit.
Whatever the output view does not cover keeps its sentinel.
"""
import numpy as np
import pytest

import oracle
from tests.util import assert_close, to_host64

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": "bfloat16", "f16": "float16", "f32": "float32"}


@pytest.fixture(scope="module")
def ta():
    import torch
    from transformer_attention_tcgen05_gb300.build import build
    build()
    import transformer_attention_tcgen05_gb300 as ta
    torch.cuda.set_device(0)
    return ta


def _dev(a: np.ndarray, dt: str):
    import torch
    return torch.from_numpy(a).cuda().to(getattr(torch, TORCH_DT[dt]))


def _check(ta, q, k, v, o, dt, family, what):
    """q, k, v, o: [B, H, N, D] views. Returns nothing; asserts parity."""
    n0 = ta.launch_count(family)
    ta.full_fwd_strided(q, k, v, o)
    assert ta.launch_count(family) > n0, f"{family} did not launch"
    assert ta.device_status() == 0
    ref = oracle.full_fwd(to_host64(q), to_host64(k), to_host64(v))
    assert_close(to_host64(o), ref, dt, what)
    import torch
    dense = ta.full_fwd(q.contiguous(), k.contiguous(), v.contiguous())
    assert torch.equal(dense, o), f"{what}: strided result differs from the contiguous one"


@pytest.mark.parametrize("dt,D,family", [("bf16", 128, "tc_flash"), ("f16", 64, "tc_flash"),
                                         ("f32", 32, "simt"), ("bf16", 32, "simt")])
def test_transposed_projection_layout(ta, dt, D, family):
    """q, k, v and o are [B, N, H, D] tensors read and written as [B, H, N, D]."""
    import torch
    B, H, Nq, Nkv = 2, 3, 300, 333
    g = np.random.default_rng(9700 + D)
    qb = _dev(g.standard_normal((B, Nq, H, D), dtype=np.float32), dt)
    kb = _dev(g.standard_normal((B, Nkv, H, D), dtype=np.float32), dt)
    vb = _dev(g.standard_normal((B, Nkv, H, D), dtype=np.float32), dt)
    ob = torch.empty_like(qb)
    q, k, v, o = (t.transpose(1, 2) for t in (qb, kb, vb, ob))
    assert not q.is_contiguous()
    _check(ta, q, k, v, o, dt, family, f"{dt} transposed D={D}")


@pytest.mark.parametrize("dt,D,family", [("bf16", 64, "tc_flash"), ("f16", 128, "tc_flash"),
                                         ("f32", 64, "simt")])
def test_packed_qkv_and_output_column_block(ta, dt, D, family):
    """q, k, v are the three slices of one [B, N, 3, H, D] projection; o is a
    column block of a [B, N, H*D + 64] buffer whose last 64 columns hold a
    sentinel the call must not touch."""
    import torch
    B, H, N = 2, 2, 257
    g = np.random.default_rng(9800 + D)
    qkv = _dev(g.standard_normal((B, N, 3, H, D), dtype=np.float32), dt)
    q, k, v = (qkv[:, :, i].transpose(1, 2) for i in range(3))
    wide = torch.full((B, N, H * D + 64), 7.0, dtype=qkv.dtype, device="cuda")
    o = wide[:, :, :H * D].unflatten(2, (H, D)).transpose(1, 2)
    assert o.stride() == (N * (H * D + 64), D, H * D + 64, 1)
    _check(ta, q, k, v, o, dt, family, f"{dt} packed qkv D={D}")
    assert (wide[:, :, H * D:] == 7.0).all(), "sentinel columns were written"


def test_broadcast_batch_of_one_ignores_its_stride(ta):
    """An extent-1 axis may carry any stride (torch reports arbitrary ones)."""
    import torch
    H, N, D = 4, 200, 64
    g = np.random.default_rng(9900)
    base = _dev(g.standard_normal((3, H, N, D), dtype=np.float32), "bf16")
    # batch stride 12345 elements (24690 bytes, not a multiple of 16) on an
    # extent-1 axis: never stepped along, so it must be accepted
    q = base[0:1].as_strided((1, H, N, D), (12345, N * D, D, 1))
    k, v = base[1:2], base[2:3]
    o = torch.empty((1, H, N, D), dtype=torch.bfloat16, device="cuda")
    _check(ta, q, k, v, o, "bf16", "tc_flash", "batch of one")


@pytest.mark.parametrize("dt,D,family", [("bf16", 128, "tc_flash"), ("f16", 64, "tc_flash"),
                                         ("f32", 64, "simt")])
def test_causal_gqa_llama_projection_layout(ta, dt, D, family):
    """Causal GQA prefill reading q from a [B, N, Hq, D] projection and k, v
    from one packed [B, N, 2, Hkv, D] projection, writing o into [B, N, Hq, D]."""
    import torch
    B, Hq, Hkv, N = 2, 4, 2, 300
    g = np.random.default_rng(9950 + D)
    qb = _dev(g.standard_normal((B, N, Hq, D), dtype=np.float32), dt)
    kvb = _dev(g.standard_normal((B, N, 2, Hkv, D), dtype=np.float32), dt)
    ob = torch.full_like(qb, 5.0)
    q, o = qb.transpose(1, 2), ob.transpose(1, 2)
    k, v = kvb[:, :, 0].transpose(1, 2), kvb[:, :, 1].transpose(1, 2)
    n0 = ta.launch_count(family)
    ta.causal_gqa_fwd_strided(q, k, v, o)
    assert ta.launch_count(family) > n0, f"{family} did not launch"
    assert ta.device_status() == 0
    ref = oracle.causal_gqa_fwd(to_host64(q), to_host64(k), to_host64(v))
    assert_close(to_host64(o), ref, dt, f"{dt} causal strided D={D}")
    dense = ta.causal_gqa_fwd(q.contiguous(), k.contiguous(), v.contiguous())
    assert torch.equal(dense, o), "strided causal result differs from the contiguous one"


@pytest.mark.parametrize("dt,B", [("bf16", 1), ("f16", 1), ("bf16", 2)])
def test_na3d_projection_layout(ta, dt, B):
    """Neighborhood attention reading q, k, v from [B, T*Hg*W, heads, D]
    projections and writing o into the same layout: a non-contiguous layout
    runs on the exact SIMT kernel, which addresses every tensor through its
    strides."""
    import torch
    grid, kernel, H, D = ((3, 20, 24), (3, 5, 7), 2, 64) if B == 1 else ((2, 8, 12), (3, 3, 5), 2, 64)
    N = grid[0] * grid[1] * grid[2]
    g = np.random.default_rng(9980 + B + len(dt))
    qb, kb, vb = (_dev(g.standard_normal((B, N, H, D), dtype=np.float32), dt) for _ in range(3))
    ob = torch.full_like(qb, 5.0)
    q, k, v, o = (t.transpose(1, 2) for t in (qb, kb, vb, ob))
    n0 = ta.launch_count("simt")
    ta.na3d_fwd_strided(q, k, v, grid, kernel, o=o)
    assert ta.launch_count("simt") > n0, "simt did not launch"
    assert ta.device_status() == 0
    ref = oracle.na3d_fwd(to_host64(q), to_host64(k), to_host64(v), grid, kernel)
    assert_close(to_host64(o), ref, dt, f"{dt} na3d strided B={B}")


def test_na3d_strided_entry_with_dense_strides_takes_the_tensor_cores(ta):
    """Contiguous tensors passed through the strided entry run the tensor-core
    kernel and give exactly the contiguous entry's result."""
    import torch
    grid, kernel, H, D = (3, 20, 24), (3, 5, 7), 2, 64
    N = grid[0] * grid[1] * grid[2]
    g = np.random.default_rng(9990)
    q, k, v = (_dev(g.standard_normal((1, H, N, D), dtype=np.float32), "bf16") for _ in range(3))
    n0 = ta.launch_count("tc_na")
    o = ta.na3d_fwd_strided(q, k, v, grid, kernel)
    assert ta.launch_count("tc_na") > n0, "tc_na did not launch"
    assert torch.equal(o, ta.na3d_fwd(q, k, v, grid, kernel))
