"""GPU parity for the ring KV cache (attn_kv_append_ring + attn_decode_gqa_ring).

A decode step -- ring append, then ring decode -- is captured once as a CUDA
graph and replayed for more than twice the cache capacity, so every row is
overwritten at least twice.  After every replay the output is checked against
the oracle's sliding-window decode over the token history (the newest
`capacity` tokens), and at the end the cache rows are checked byte for byte
against the ring layout (token t in row t % capacity, the newest such token).
"""
import numpy as np
import pytest

import oracle
from tests.util import assert_close, to_dev, to_host64
from workloads import draw, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ta():
    import torch
    from transformer_attention_tcgen05_gb300.build import build
    build()
    import transformer_attention_tcgen05_gb300 as ta
    torch.cuda.set_device(0)
    return ta


@pytest.mark.parametrize("dt,Hq,Hkv,D,cap,prefill", [("bf16", 8, 2, 128, 100, (0, 37)),
                                                     ("f16", 4, 4, 64, 33, (5, 20))])
def test_ring_decode_step_replayed_past_capacity(ta, dt, Hq, Hkv, D, cap, prefill):
    import torch
    B = 2
    steps = 2 * cap + 30
    T = max(prefill) + steps
    rng = np.random.Generator(np.random.PCG64(8700 + cap))
    k_hist = draw(rng, (B, Hkv, T, D), dt)       # every token each sequence will hold
    v_hist = draw(rng, (B, Hkv, T, D), dt)
    k64, v64 = to_f64(k_hist, dt), to_f64(v_hist, dt)
    n = np.array(prefill, dtype=np.int64)

    # the cache after the prefill tokens, in ring rows (t % cap)
    kc_h = np.zeros((B, Hkv, cap, D), dtype=k_hist.dtype)
    vc_h = np.zeros_like(kc_h)
    for b in range(B):
        for t in range(n[b]):
            kc_h[b, :, t % cap] = k_hist[b, :, t]
            vc_h[b, :, t % cap] = v_hist[b, :, t]
    kc, vc = to_dev(kc_h, dt), to_dev(vc_h, dt)
    sl = torch.from_numpy(n.astype(np.int32)).cuda()
    q = to_dev(np.zeros((B, Hq, D), dtype=k_hist.dtype), dt)
    kn = to_dev(np.zeros((B, Hkv, D), dtype=k_hist.dtype), dt)
    vn = to_dev(np.zeros((B, Hkv, D), dtype=k_hist.dtype), dt)
    o = torch.empty_like(q)
    ws = torch.zeros(ta.decode_workspace_bytes(B, Hq, Hkv, cap, D), dtype=torch.uint8,
                     device="cuda")

    # first calls outside the capture (per-device set-up of the library)
    sl_w, kc_w, vc_w = sl.clone(), kc.clone(), vc.clone()
    ta.kv_append_ring(kc_w, vc_w, kn, vn, sl_w)
    ta.decode_gqa_ring(q, kc_w, vc_w, sl_w, o=o, workspace=ws)
    torch.cuda.synchronize()
    assert ta.device_status() == 0

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ta.kv_append_ring(kc, vc, kn, vn, sl)
        ta.decode_gqa_ring(q, kc, vc, sl, o=o, workspace=ws)
    for step in range(steps):
        qh = draw(rng, (B, Hq, D), dt)
        q.copy_(to_dev(qh, dt))
        kn.copy_(to_dev(np.ascontiguousarray(k_hist[np.arange(B), :, n]), dt))
        vn.copy_(to_dev(np.ascontiguousarray(v_hist[np.arange(B), :, n]), dt))
        g.replay()
        n += 1
        torch.cuda.synchronize()
        assert sl.tolist() == n.tolist()
        ref = oracle.decode_ring(to_f64(qh, dt), k64, v64, n, cap)
        assert_close(to_host64(o), ref, dt, f"ring decode step {step} (n = {n.tolist()})")
    assert ta.device_status() == 0

    # ring layout: row r holds the newest token t < n with t % cap == r
    want_k = np.zeros_like(kc_h)
    want_v = np.zeros_like(vc_h)
    for b in range(B):
        for r in range(cap):
            t = r + ((n[b] - 1 - r) // cap) * cap
            want_k[b, :, r] = k_hist[b, :, t]
            want_v[b, :, r] = v_hist[b, :, t]
    got_k = kc.cpu().view(torch.int16).numpy().view(np.uint16)
    got_v = vc.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got_k, want_k.view(np.uint16)), "K ring rows"
    assert np.array_equal(got_v, want_v.view(np.uint16)), "V ring rows"


def test_linear_decode_still_rejects_a_length_past_capacity(ta):
    """The linear entry keeps its bound: seq_len > Lmax is a device check
    (reported, output untouched); the ring entry accepts the same length."""
    import torch
    B, Hq, Hkv, L, D = 1, 4, 1, 64, 64
    rng = np.random.Generator(np.random.PCG64(8800))
    kc_h, vc_h = draw(rng, (B, Hkv, L, D), "bf16"), draw(rng, (B, Hkv, L, D), "bf16")
    qh = draw(rng, (B, Hq, D), "bf16")
    kc, vc, q = to_dev(kc_h, "bf16"), to_dev(vc_h, "bf16"), to_dev(qh, "bf16")
    sl = torch.tensor([L + 5], dtype=torch.int32, device="cuda")
    o = torch.full_like(q, 3.0)
    ta.decode_gqa(q, kc, vc, sl, o=o)
    assert ta.device_status() == 6          # ATTN_ERR_DEVICE_CHECK
    assert (o == 3.0).all()
    o = ta.decode_gqa_ring(q, kc, vc, sl)
    assert ta.device_status() == 0
    ref = oracle.decode_gqa(to_f64(qh, "bf16"), to_f64(kc_h, "bf16"), to_f64(vc_h, "bf16"), [L])
    assert_close(to_host64(o), ref, "bf16", "ring decode of a wrapped full cache")
