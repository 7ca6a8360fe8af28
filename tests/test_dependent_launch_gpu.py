"""Programmatic dependent launches read what the kernel before them wrote.

Decode and the tcgen05 attention kernel are launched as programmatic
dependents of the previous kernel on the stream, and the neighborhood kernel
lets the kernel behind it start launching at entry.  A dependent's CTAs can
therefore be resident while the previous kernel still runs; they must wait
for it before any global access.  Here a small neighborhood problem (a few
dozen CTAs, so most SMs are free for the dependent) writes its output into a
buffer filled with NaN, and the kernel launched right behind it on the same
stream, with nothing in between, takes its queries from that buffer.  A
dependent that read too early would see NaN or stale rows; the oracle on the
queries as finally written decides.
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


def _neighborhood_output_buffer(ta, seed):
    """A NaN-filled buffer and a neighborhood call (4 heads of a 3 x 9 x 40
    grid, 48 boxes on 24 CTAs) that will write it."""
    import torch
    w = WORKLOADS["na3d_21x60x104_k11"].with_(grid=(3, 9, 40), kernel=(5, 3, 9), H=4, N=3 * 9 * 40,
                                             seed=seed)
    x = make_inputs(w)
    q, k, v = (to_dev(x[c], "bf16") for c in "qkv")
    o = torch.full_like(q, float("nan"))
    return o, lambda: ta.na3d_fwd(q, k, v, w.grid, w.kernel, o=o)


def test_decode_reads_queries_the_neighborhood_kernel_just_wrote(ta):
    import torch
    o, run_na = _neighborhood_output_buffer(ta, 7811)
    w = WORKLOADS["gqa_decode"].with_(B=2, Lmax=600, seq_len=(600, 311), seed=7812)
    x = make_inputs(w)
    kc, vc = to_dev(x["k"], "bf16"), to_dev(x["v"], "bf16")
    sl = torch.from_numpy(x["seq_len"]).cuda()
    ws = torch.zeros(ta.decode_workspace_bytes(w.B, w.H, w.Hkv, w.Lmax, w.D), dtype=torch.uint8,
                     device="cuda")
    dq = o.view(-1)[:w.B * w.H * w.D].view(w.B, w.H, w.D)      # a view: no launch in between
    od = torch.empty_like(dq)
    torch.cuda.synchronize()
    n_na, n_dec = ta.launch_count("tc_na"), ta.launch_count("decode")
    run_na()
    ta.decode_gqa(dq, kc, vc, sl, o=od, workspace=ws)
    torch.cuda.synchronize()
    assert ta.launch_count("tc_na") > n_na and ta.launch_count("decode") > n_dec
    qh = to_host64(dq)
    assert np.isfinite(qh).all()
    ref = oracle.decode_gqa(qh, to_f64(x["k"], "bf16"), to_f64(x["v"], "bf16"), x["seq_len"])
    assert_close(to_host64(od), ref, "bf16", "decode behind the neighborhood kernel")
    assert ta.device_status() == 0


def test_attention_reads_queries_the_neighborhood_kernel_just_wrote(ta):
    import torch
    o, run_na = _neighborhood_output_buffer(ta, 7821)
    B, H, N, D = o.shape                                         # [1, 4, 1080, 64]
    w = WORKLOADS["na3d_21x60x104_k11"].with_(grid=(3, 9, 40), kernel=(5, 3, 9), H=H, N=N, seed=7822)
    x = make_inputs(w)
    k, v = to_dev(x["k"], "bf16"), to_dev(x["v"], "bf16")
    oa = torch.empty_like(o)
    torch.cuda.synchronize()
    n_na, n_tc = ta.launch_count("tc_na"), ta.launch_count("tc_flash")
    run_na()
    ta.full_fwd(o, k, v, o=oa)
    torch.cuda.synchronize()
    assert ta.launch_count("tc_na") > n_na and ta.launch_count("tc_flash") > n_tc
    qh = to_host64(o)
    assert np.isfinite(qh).all()
    ref = oracle.full_fwd(qh, to_f64(x["k"], "bf16"), to_f64(x["v"], "bf16"))
    assert_close(to_host64(oa), ref, "bf16", "attention behind the neighborhood kernel")
    assert ta.device_status() == 0
