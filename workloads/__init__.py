"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds no attention arithmetic: it only draws random tensors, rounds
them to the storage dtype and lays out position ids.  Both the CUDA path and the
CPU oracle consume the exact host arrays produced here, so input rounding never
counts as error on either side.

Recipe (fixed, so every run sees the same numbers):
  * numpy ``Generator(PCG64(seed))``, ``standard_normal`` in float32;
  * draws in the order Q, K, V (decode: q, k_cache, v_cache);
  * bf16 storage is the round-to-nearest-even of that float32 draw, kept as the
    raw uint16 bit pattern;
  * the seed of workload ``c`` (1-based, in the order of ``WORKLOADS``) is
    ``1000 + c``; a variant adds ``100 * k``.

The shapes follow the workloads of the attention pages: tiny full MHA,
neighborhood-attention clamp cases (candle NA3D PR, "kernel exceeds grid
extent" commit), Llama-style GQA decode over a device-resident KV cache (fak
GPU.md section 0) and FLUX joint text+image attention with a 4-axis RoPE
(iris.c issue #15, the GGML lessons list, item 3).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import numpy as np

__all__ = [
    "bf16_round", "bf16_to_f32", "draw", "flux_positions", "Workload", "WORKLOADS",
    "make_inputs",
]


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern (uint16), round to nearest, ties to even.

    Inputs are finite standard-normal draws; NaN/Inf are not expected but are
    kept NaN/Inf (the exponent field is untouched by the carry for them only
    when the mantissa is already saturated, which cannot occur for N(0,1)).
    """
    a = np.ascontiguousarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    return r.reshape(a.shape)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit pattern (uint16) -> float32 (exact widening)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).reshape(b.shape)


def draw(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """One N(0,1) tensor: float32 for 'f32', uint16 bf16 bits for 'bf16',
    float16 (round to nearest even of the float32 draw) for 'f16'."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return bf16_round(x)
    if dtype == "f16":
        return x.astype(np.float16)
    raise ValueError(f"unknown dtype {dtype!r}")


def flux_positions(n_txt: int, rows: int, cols: int) -> np.ndarray:
    """Position ids [N, 4] int32 for a text-first joint sequence.

    Text token j gets (0, 0, 0, j); image token r*cols + c gets (0, r, c, 0).
    The text block comes first in the concatenation (the reading taken for the
    FLUX joint-attention workload: "512 text + 4096 image tokens").
    """
    n = n_txt + rows * cols
    pos = np.zeros((n, 4), dtype=np.int32)
    pos[:n_txt, 3] = np.arange(n_txt, dtype=np.int32)
    r, c = np.meshgrid(np.arange(rows, dtype=np.int32), np.arange(cols, dtype=np.int32),
                       indexing="ij")
    pos[n_txt:, 1] = r.reshape(-1)
    pos[n_txt:, 2] = c.reshape(-1)
    return pos


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload.  ``kind`` selects the entry point."""
    name: str
    kind: str                 # "full" | "na3d" | "decode" | "joint"
    dtype: str                # "f32" | "bf16" | "f16"
    seed: int
    B: int = 1
    H: int = 1                # heads (query heads for decode)
    N: int = 0                # tokens (full / joint / na3d: T*Hg*W)
    D: int = 32
    grid: Optional[Tuple[int, int, int]] = None      # na3d (T, Hg, W)
    kernel: Optional[Tuple[int, int, int]] = None    # na3d requested kernel
    Hkv: int = 0              # decode
    Lmax: int = 0             # decode capacity
    seq_len: Optional[Tuple[int, ...]] = None        # decode; None = all Lmax
    n_txt: int = 0            # joint
    img: Optional[Tuple[int, int]] = None            # joint (rows, cols)
    axes_dim: Tuple[int, int, int, int] = (32, 32, 32, 32)
    theta: float = 10000.0

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _na(name, dtype, seed, grid, kernel, heads, D, B=1):
    t, h, w = grid
    return Workload(name=name, kind="na3d", dtype=dtype, seed=seed, B=B, H=heads,
                    N=t * h * w, D=D, grid=tuple(grid), kernel=tuple(kernel))


#: The five workloads (seed 1000 + position, 1-based; bf16 variants add 100).
WORKLOADS: Dict[str, Workload] = {
    # 1. tiny full MHA, fp32
    "mha_tiny": Workload("mha_tiny", "full", "f32", 1001, B=1, H=2, N=64, D=32),
    # 2. neighborhood-attention clamp cases, fp32 and bf16
    "na3d_1x4x4_k3x7x7_f32": _na("na3d_1x4x4_k3x7x7_f32", "f32", 1002, (1, 4, 4), (3, 7, 7), 4, 32),
    "na3d_1x4x4_k3x7x7_bf16": _na("na3d_1x4x4_k3x7x7_bf16", "bf16", 1102, (1, 4, 4), (3, 7, 7), 4, 32),
    "na3d_9x64x64_k11_f32": _na("na3d_9x64x64_k11_f32", "f32", 1202, (9, 64, 64), (11, 11, 11), 4, 32),
    "na3d_9x64x64_k11_bf16": _na("na3d_9x64x64_k11_bf16", "bf16", 1302, (9, 64, 64), (11, 11, 11), 4, 32),
    # 3. Llama-style GQA decode, bf16 cache
    "gqa_decode": Workload("gqa_decode", "decode", "bf16", 1003, B=8, H=32, D=128, Hkv=8,
                           Lmax=4096),
    # 4. FLUX joint attention with 4-axis RoPE, bf16
    "flux_joint": Workload("flux_joint", "joint", "bf16", 1004, B=1, H=24, N=4608, D=128,
                           n_txt=512, img=(64, 64)),
    # 5. large 3D neighborhood attention, bf16
    "na3d_21x60x104_k11": _na("na3d_21x60x104_k11", "bf16", 1005, (21, 60, 104), (11, 11, 11), 8, 64),
}


def make_inputs(w: Workload) -> Dict[str, np.ndarray]:
    """Host arrays for workload ``w``.

    Returns q, k, v (storage dtype: float32 or uint16 bf16 bits) in the
    heads-major layout [B, H, N, D] (decode: q [B, Hq, D], k/v [B, Hkv, Lmax, D],
    plus ``seq_len`` int32 [B]); joint workloads add ``pos`` int32 [N, 4].
    """
    rng = np.random.Generator(np.random.PCG64(w.seed))
    out: Dict[str, np.ndarray] = {}
    if w.kind == "decode":
        out["q"] = draw(rng, (w.B, w.H, w.D), w.dtype)
        out["k"] = draw(rng, (w.B, w.Hkv, w.Lmax, w.D), w.dtype)
        out["v"] = draw(rng, (w.B, w.Hkv, w.Lmax, w.D), w.dtype)
        sl = w.seq_len if w.seq_len is not None else (w.Lmax,) * w.B
        out["seq_len"] = np.asarray(sl, dtype=np.int32)
        return out
    shape = (w.B, w.H, w.N, w.D)
    out["q"] = draw(rng, shape, w.dtype)
    out["k"] = draw(rng, shape, w.dtype)
    out["v"] = draw(rng, shape, w.dtype)
    if w.kind == "joint":
        rows, cols = w.img
        out["pos"] = flux_positions(w.n_txt, rows, cols)
        assert out["pos"].shape[0] == w.N
    return out


def to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of a storage array to float64."""
    if dtype == "bf16":
        return bf16_to_f32(x).astype(np.float64)
    return np.asarray(x, dtype=np.float32).astype(np.float64)
