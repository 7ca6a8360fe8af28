"""Launch one entry point on a seeded synthetic workload, for profilers.

    python -m transformer_attention_tcgen05_gb300.profile_case KERNEL
        [--frames T] [--warmup W] [--launches N]

KERNEL is one of:
  joint   FLUX joint attention with 4-axis RoPE: B 1, 24 heads, 512 text +
          64 x 64 image tokens, D 128 (attn_rope_joint_fwd)
  na3d    3D neighborhood attention, 21 x 60 x 104 grid, 11^3 window,
          8 heads, D 64 (attn_na3d_fwd); --frames shrinks the T axis
  decode  GQA decode, B 8, 32 query / 8 KV heads, 4096 cached rows, D 128
          (attn_decode_gqa)
  causal  causal GQA prefill, B 1, 32 query / 8 KV heads, 4096 tokens, D 128
          (attn_causal_gqa_fwd)

The inputs are the benchmark's seeded bf16 draws.  W untimed launches run
first, then N more; the process exits non-zero if the device reports an
error.  Nothing is timed here: a profiler (ncu -k / -s / -c) picks the
launches it wants from this fixed sequence.
"""
import argparse
import sys

import numpy as np
import torch

import transformer_attention_tcgen05_gb300 as ta
from workloads import WORKLOADS, make_inputs


def _dev(x, dev):
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev)


def build_case(kernel: str, frames: int, dev):
    """Return a zero-argument callable that launches `kernel` once."""
    if kernel == "joint":
        w = WORKLOADS["flux_joint"]
        h = make_inputs(w)
        q, k, v = (_dev(h[n], dev) for n in "qkv")
        pos = torch.from_numpy(h["pos"]).to(dev)
        o = torch.empty_like(q)
        ws = torch.empty(ta.rope_joint_workspace_bytes(w.B, w.H, w.N, w.D, torch.bfloat16),
                         dtype=torch.uint8, device=dev)
        return lambda: ta.rope_joint_fwd(q, k, v, pos, w.axes_dim, w.theta, o=o, workspace=ws)
    if kernel == "na3d":
        w = WORKLOADS["na3d_21x60x104_k11"]
        if frames:
            _, hg, wd = w.grid
            w = w.with_(grid=(frames, hg, wd), N=frames * hg * wd)
        h = make_inputs(w)
        q, k, v = (_dev(h[n], dev) for n in "qkv")
        o = torch.empty_like(q)
        return lambda: ta.na3d_fwd(q, k, v, w.grid, w.kernel, o=o)
    if kernel == "decode":
        w = WORKLOADS["gqa_decode"]
        h = make_inputs(w)
        q, kc, vc = (_dev(h[n], dev) for n in "qkv")
        sl = torch.from_numpy(h["seq_len"]).to(dev)
        o = torch.empty_like(q)
        ws = torch.zeros(ta.decode_workspace_bytes(w.B, w.H, w.Hkv, w.Lmax, w.D),
                         dtype=torch.uint8, device=dev)
        return lambda: ta.decode_gqa(q, kc, vc, sl, o=o, workspace=ws)
    if kernel == "causal":
        g = torch.Generator(device="cpu").manual_seed(1006)
        q = torch.randn(1, 32, 4096, 128, generator=g).bfloat16().to(dev)
        k = torch.randn(1, 8, 4096, 128, generator=g).bfloat16().to(dev)
        v = torch.randn(1, 8, 4096, 128, generator=g).bfloat16().to(dev)
        o = torch.empty_like(q)
        return lambda: ta.causal_gqa_fwd(q, k, v, o=o)
    raise SystemExit(f"unknown kernel {kernel!r}")


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("kernel", choices=["joint", "na3d", "decode", "causal"])
    ap.add_argument("--frames", type=int, default=0, help="na3d: T extent (default 21)")
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--launches", type=int, default=1)
    a = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    run = build_case(a.kernel, a.frames, dev)
    for _ in range(a.warmup + a.launches):
        run()
    torch.cuda.synchronize()
    st = ta.device_status()
    print(f"{a.kernel}: {a.warmup} + {a.launches} launches, device status {st}")
    return 0 if st == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
