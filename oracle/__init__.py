"""fp64 CPU oracle for scaled-dot-product attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import this package.  The CUDA library never does, and this
package never imports the CUDA library: the two share only the seeded input
generators of ``workloads``.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, OpenMP
over query rows); this module only marshals numpy arrays.  Inputs are float64
arrays (exact widenings of the float32 / bf16 host arrays), layouts as in the
C file:  full / joint / na3d  q, k, v [B, H, N, D];  decode q [B, Hq, D],
k, v [B, Hkv, Lmax, D].  ``scale=None`` means 1/sqrt(D).

Pins (checked by ``tests/test_oracle_*.py``, all on the CPU):
  * brute force with an independent window characterisation on tiny inputs;
  * torch's float64 CPU scaled_dot_product_attention (with a boolean mask);
  * invariants (rows sum to 1, constant V, Q = 0, k >= extent == full,
    decode == full with Nq = 1, RoPE norm / identity / relative shift,
    ring decode: a one-row ring returns the newest V, tokens older than the
    window do not matter, a ring at least as long as the history is decode);
  * the pages' clamp cases and hand-computed window starts (tests/golden).
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

import numpy as np

from .build import build_oracle

_LIB = None

_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_vp = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_d = ctypes.c_double


def lib():
    """Load (building first if needed) liboracle.so."""
    global _LIB
    if _LIB is None:
        path = os.environ.get("ATTN_ORACLE_LIB") or build_oracle()
        L = ctypes.CDLL(path)
        L.oracle_max_threads.restype = _i
        L.oracle_full_fwd.argtypes = [_f64p, _f64p, _f64p, _f64p, _vp, _i, _i, _i, _i, _i, _d, _i]
        L.oracle_full_rows.argtypes = [_f64p, _f64p, _f64p, _f64p, _i, _i, _i, _i, _i, _d,
                                       _i64p, _i64, _i]
        L.oracle_rope_rotate.argtypes = [_f64p, _i32p, _i, _i, _i, _i32p, _d]
        L.oracle_joint_fwd.restype = _i
        L.oracle_joint_fwd.argtypes = [_f64p, _f64p, _f64p, _f64p, _i, _i, _i, _i, _i32p, _i32p,
                                       _d, _d, _vp, _i64, _i]
        L.oracle_decode_gqa.argtypes = [_f64p, _f64p, _f64p, _i32p, _f64p, _i, _i, _i, _i, _i,
                                        _d, _i]
        L.oracle_causal_gqa_fwd.argtypes = [_f64p, _f64p, _f64p, _f64p, _i, _i, _i, _i, _i, _d,
                                            _vp, _i64, _i]
        L.oracle_na_window_start.restype = _i
        L.oracle_na_window_start.argtypes = [_i, _i, _i]
        L.oracle_na3d_window_starts.argtypes = [_i, _i, _i, _i32p, _i32p]
        L.oracle_na3d_fwd.argtypes = [_f64p, _f64p, _f64p, _f64p, _vp, _i, _i, _i, _i, _i, _i,
                                      _i32p, _d, _vp, _i64, _i]
        _LIB = L
    return _LIB


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def _c(x, dt=np.float64):
    return np.ascontiguousarray(x, dtype=dt)


def _scale(scale: Optional[float], D: int) -> float:
    return 1.0 / math.sqrt(D) if scale is None or scale <= 0 else float(scale)


def full_fwd(q, k, v, scale=None, return_p=False, threads=0):
    """Full attention. q [B,H,Nq,D], k/v [B,H,Nkv,D] -> o (and p [B,H,Nq,Nkv])."""
    q, k, v = _c(q), _c(k), _c(v)
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    assert k.shape == (B, H, Nkv, D) and v.shape == k.shape
    o = np.empty_like(q)
    p = np.empty((B, H, Nq, Nkv)) if return_p else None
    lib().oracle_full_fwd(q, k, v, o, p.ctypes.data if return_p else None,
                          B, H, Nq, Nkv, D, _scale(scale, D), threads)
    return (o, p) if return_p else o


def full_rows(q, k, v, rows: Sequence[int], scale=None, threads=0):
    """Full attention on flattened query rows (b*H*Nq + h*Nq + i) -> [len(rows), D]."""
    q, k, v = _c(q), _c(k), _c(v)
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    r = _c(rows, np.int64)
    o = np.empty((r.size, D))
    lib().oracle_full_rows(q, k, v, o, B, H, Nq, Nkv, D, _scale(scale, D), r, r.size, threads)
    return o


def rope_rotate(x, pos, axes_dim=(32, 32, 32, 32), theta=10000.0):
    """Rotated copy of x [B,H,N,D] (multi-axis RoPE on adjacent pairs)."""
    x = _c(x).copy()
    B, H, N, D = x.shape
    ax = _c(axes_dim, np.int32)
    assert int(ax.sum()) == D and all(a % 2 == 0 for a in ax)
    lib().oracle_rope_rotate(x, _c(pos, np.int32), B * H, N, D, ax, float(theta))
    return x


def joint_fwd(q, k, v, pos, axes_dim=(32, 32, 32, 32), theta=10000.0, scale=None,
              rows: Optional[Sequence[int]] = None, threads=0):
    """RoPE on q and k, then full attention over the joint sequence."""
    q, k, v = _c(q), _c(k), _c(v)
    B, H, N, D = q.shape
    ax = _c(axes_dim, np.int32)
    assert int(ax.sum()) == D and all(a % 2 == 0 for a in ax)
    pos = _c(pos, np.int32)
    assert pos.shape == (N, 4)
    r = None if rows is None else _c(rows, np.int64)
    o = np.empty_like(q) if r is None else np.empty((r.size, D))
    err = lib().oracle_joint_fwd(q, k, v, o, B, H, N, D, pos, ax, float(theta),
                                 _scale(scale, D), None if r is None else r.ctypes.data,
                                 0 if r is None else r.size, threads)
    if err:
        raise MemoryError("oracle_joint_fwd: out of host memory")
    return o


def decode_gqa(q, kc, vc, seq_len, scale=None, threads=0):
    """GQA decode: q [B,Hq,D], k/v cache [B,Hkv,Lmax,D], seq_len [B] -> o [B,Hq,D]."""
    q, kc, vc = _c(q), _c(kc), _c(vc)
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = kc.shape
    assert Hq % Hkv == 0
    sl = _c(seq_len, np.int32)
    assert sl.shape == (B,) and np.all((sl >= 1) & (sl <= Lmax))
    o = np.empty_like(q)
    lib().oracle_decode_gqa(q, kc, vc, sl, o, B, Hq, Hkv, Lmax, D, _scale(scale, D), threads)
    return o


def decode_ring(q, k_tokens, v_tokens, n_tokens, capacity, scale=None, threads=0):
    """Decode over a ring KV cache of `capacity` rows, stated on the token
    history: k_tokens / v_tokens [B, Hkv, T, D] hold every token appended to
    each sequence in order, n_tokens [B] how many were appended (1 <= n <= T).
    A ring of `capacity` rows keeps the most recent `capacity` of them, so
    query b attends to tokens [max(0, n_b - capacity), n_b): a sliding window
    (fak "GPU - the in-kernel forward pass", section 3b: a dynamic / ring
    device KV as the follow-up to the fixed-capacity one).  The window is
    gathered in time order into a cache and handed to the pinned decode."""
    q, k_tokens, v_tokens = _c(q), _c(k_tokens), _c(v_tokens)
    B, Hkv, T, D = k_tokens.shape
    n = np.asarray(n_tokens, dtype=np.int64)
    assert n.shape == (B,) and np.all((n >= 1) & (n <= T)) and capacity >= 1
    L = int(min(capacity, n.max()))
    kc = np.zeros((B, Hkv, L, D))
    vc = np.zeros((B, Hkv, L, D))
    lens = np.empty(B, dtype=np.int32)
    for b in range(B):
        lo = max(0, int(n[b]) - capacity)
        lens[b] = int(n[b]) - lo
        kc[b, :, :lens[b]] = k_tokens[b, :, lo:n[b]]
        vc[b, :, :lens[b]] = v_tokens[b, :, lo:n[b]]
    return decode_gqa(q, kc, vc, lens, scale=scale, threads=threads)


def causal_gqa_fwd(q, k, v, scale=None, rows: Optional[Sequence[int]] = None, threads=0):
    """Causal GQA prefill: q [B,Hq,N,D], k/v [B,Hkv,N,D]; query i sees keys j <= i."""
    q, k, v = _c(q), _c(k), _c(v)
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    assert k.shape == (B, Hkv, N, D) and v.shape == k.shape and Hq % Hkv == 0
    r = None if rows is None else _c(rows, np.int64)
    o = np.empty_like(q) if r is None else np.empty((r.size, D))
    lib().oracle_causal_gqa_fwd(q, k, v, o, B, Hq, Hkv, N, D, _scale(scale, D),
                                None if r is None else r.ctypes.data, 0 if r is None else r.size,
                                threads)
    return o


def na_window_start(i: int, n: int, k: int) -> int:
    return int(lib().oracle_na_window_start(i, n, k))


def na3d_window_starts(grid, kernel):
    """int32 [T*Hg*W, 3]: per-query (t, h, w) window starts."""
    T, Hg, W = grid
    out = np.empty((T * Hg * W, 3), dtype=np.int32)
    lib().oracle_na3d_window_starts(T, Hg, W, _c(kernel, np.int32), out)
    return out


def na3d_fwd(q, k, v, grid, kernel, scale=None, rows: Optional[Sequence[int]] = None,
             return_p=False, threads=0):
    """3D neighborhood attention; q/k/v [B,H,T*Hg*W,D]."""
    q, k, v = _c(q), _c(k), _c(v)
    B, H, N, D = q.shape
    T, Hg, W = grid
    assert N == T * Hg * W
    kern = _c(kernel, np.int32)
    assert kern.shape == (3,) and np.all((kern > 0) & (kern % 2 == 1))
    p = None
    if rows is None:
        o = np.empty_like(q)
        if return_p:
            p = np.empty((B, H, N, N))
        lib().oracle_na3d_fwd(q, k, v, o, p.ctypes.data if p is not None else None,
                              B, H, T, Hg, W, D, kern, _scale(scale, D), None, 0, threads)
    else:
        r = _c(rows, np.int64)
        o = np.empty((r.size, D))
        lib().oracle_na3d_fwd(q, k, v, o, None, B, H, T, Hg, W, D, kern, _scale(scale, D),
                              r.ctypes.data, r.size, threads)
    return (o, p) if return_p else o
