"""Python binding of libattn (include/libattn.h) -- argument marshalling only.

Every step of the attention path runs in the CUDA library; this module checks
tensor arguments, allocates outputs with PyTorch (PyTorch provides device
memory and streams, nothing else) and calls the C ABI through ctypes on the
current CUDA stream.  There is no fallback: if the library is not built, or
the tensors are not on a CUDA device, calls raise.

Entry points (names as in the C ABI, without the ``attn_`` prefix):
    full_fwd(q, k, v)                          q, k, v [B, H, N, D]
    rope_joint_fwd(q, k, v, pos, axes_dim, theta)
    decode_gqa(q, k_cache, v_cache, seq_len)   q [B, Hq, D], caches [B, Hkv, Lmax, D]
    na3d_fwd(q, k, v, grid, kernel)            q, k, v [B, heads, T*Hg*W, D]
    na3d_window_starts(grid, kernel)
    kv_append(k_cache, v_cache, k_new, v_new, seq_len)   device-side position, graph-stable
    causal_gqa_fwd(q, k, v)                    q [B, Hq, N, D], k/v [B, Hkv, N, D], causal
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

__all__ = [
    "AttnError", "lib", "full_fwd", "full_fwd_strided", "causal_gqa_fwd_strided", "na3d_fwd_strided", "rope_joint_fwd", "decode_gqa", "na3d_fwd", "causal_gqa_fwd",
    "na3d_window_starts", "kv_append", "kv_append_ring", "decode_gqa_ring", "decode_workspace_bytes", "rope_joint_workspace_bytes",
    "device_status", "debug_wait_test", "launch_count", "version", "FAMILIES", "LIB_PATH",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libattn.so")

ATTN_F32, ATTN_BF16, ATTN_F16 = 0, 1, 2
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration",
          3: "insufficient resources", 4: "CUDA error", 5: "device wait timed out",
          6: "device-side check failed"}
#: kernel families of attn_launch_count
FAMILIES = {"simt": 0, "tc_flash": 1, "decode": 2, "rope": 3, "na_starts": 4, "tc_na": 5,
            "kv_append": 6, "debug": 7}


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, 'unknown status')} (status {status})")


_lib = None
_vp, _i, _f, _sz, _u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64


def lib() -> ctypes.CDLL:
    """The loaded libattn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libattn is not built ({LIB_PATH} missing): run "
                               "`python -m transformer_attention_tcgen05_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        L.attn_full_fwd.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp]
        L.attn_rope_joint_fwd.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp,
                                          ctypes.POINTER(_i), _f, _i, _f, _vp, _sz, _vp]
        L.attn_rope_joint_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
        L.attn_rope_joint_workspace_bytes.restype = _sz
        L.attn_decode_gqa.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp,
                                      _sz, _vp]
        L.attn_decode_gqa_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
        L.attn_decode_gqa_workspace_bytes.restype = _sz
        L.attn_na3d_fwd.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                                    ctypes.POINTER(_i), _i, _f, _vp]
        L.attn_na3d_window_starts.argtypes = [_i, _i, _i, ctypes.POINTER(_i), _vp, _vp]
        L.attn_kv_append.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp]
        L.attn_kv_append_ring.argtypes = L.attn_kv_append.argtypes
        L.attn_decode_gqa_ring.argtypes = L.attn_decode_gqa.argtypes
        L.attn_causal_gqa_fwd.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp]
        _st = ctypes.POINTER(ctypes.c_int64)
        L.attn_full_fwd_strided.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                            _st, _st, _st, _st, _i, _f, _vp]
        L.attn_causal_gqa_fwd_strided.argtypes = L.attn_full_fwd_strided.argtypes
        L.attn_na3d_fwd_strided.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                                            ctypes.POINTER(_i), _st, _st, _st, _st, _i, _f, _vp]
        L.attn_status_string.argtypes = [_i]
        L.attn_status_string.restype = ctypes.c_char_p
        L.attn_device_status.argtypes = [_vp]
        L.attn_debug_wait_test.argtypes = [_u64, _vp]
        L.attn_launch_count.argtypes = [_i]
        L.attn_launch_count.restype = _u64
        L.attn_version.restype = ctypes.c_char_p
        for name in ("attn_full_fwd", "attn_rope_joint_fwd", "attn_decode_gqa", "attn_na3d_fwd",
                     "attn_na3d_window_starts", "attn_device_status", "attn_kv_append",
                     "attn_causal_gqa_fwd", "attn_full_fwd_strided", "attn_kv_append_ring",
                     "attn_causal_gqa_fwd_strided", "attn_na3d_fwd_strided",
                     "attn_decode_gqa_ring"):
            getattr(L, name).restype = _i
        _lib = L
    return _lib


def _check(st: int, where: str):
    if st != 0:
        raise AttnError(st, where)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return ATTN_F32
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float16:
        return ATTN_F16
    raise TypeError(f"unsupported dtype {t.dtype} (float32, bfloat16 or float16)")


def _cuda(*ts: torch.Tensor, strided: bool = False):
    dev = ts[0].device
    for t in ts:
        if not t.is_cuda:
            raise ValueError("libattn tensors must be on a CUDA device")
        if t.device != dev:
            raise ValueError("all tensors must be on the same device")
        if not strided and not t.is_contiguous():
            raise ValueError("libattn tensors must be contiguous")
    return dev


def _stream(dev) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _ints(vals: Sequence[int], n: int):
    vals = [int(x) for x in vals]
    if len(vals) != n:
        raise ValueError(f"expected {n} integers, got {len(vals)}")
    return (_i * n)(*vals)


def _scale(scale: Optional[float]) -> float:
    return 0.0 if scale is None else float(scale)


def full_fwd(q, k, v, o=None, scale=None):
    """Full attention; q [B,H,Nq,D], k/v [B,H,Nkv,D] -> o [B,H,Nq,D]."""
    dev = _cuda(q, k, v)
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    if k.shape != (B, H, Nkv, D) or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k/v must be [B, H, Nkv, D] with q's dtype")
    o = torch.empty_like(q) if o is None else o
    _cuda(q, o)
    with torch.cuda.device(dev):
        _check(lib().attn_full_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   B, H, Nq, Nkv, D, _dtype(q), _scale(scale), _stream(dev)),
               "attn_full_fwd")
    return o


def _strides(t):
    if t.stride(-1) != 1:
        raise ValueError("the last (D) dimension must be contiguous")
    return (ctypes.c_int64 * 3)(*t.stride()[:3])


def full_fwd_strided(q, k, v, o=None, scale=None):
    """Full attention on strided [B,H,N,D] views (D contiguous), read and
    written in place: e.g. q.transpose(1, 2) of a [B,N,H,D] projection or
    slices of a packed QKV tensor. o defaults to a new contiguous tensor."""
    dev = _cuda(q, k, v, strided=True)
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    if k.shape != (B, H, Nkv, D) or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k/v must be [B, H, Nkv, D] with q's dtype")
    o = torch.empty(q.shape, dtype=q.dtype, device=q.device) if o is None else o
    _cuda(q, o, strided=True)
    if o.shape != q.shape or o.dtype != q.dtype:
        raise ValueError("o must be [B, H, Nq, D] with q's dtype")
    with torch.cuda.device(dev):
        _check(lib().attn_full_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                           B, H, Nq, Nkv, D, _strides(q), _strides(k),
                                           _strides(v), _strides(o), _dtype(q), _scale(scale),
                                           _stream(dev)),
               "attn_full_fwd_strided")
    return o


def causal_gqa_fwd(q, k, v, o=None, scale=None):
    """Causal GQA prefill: q [B,Hq,N,D], k/v [B,Hkv,N,D] -> o [B,Hq,N,D]."""
    dev = _cuda(q, k, v)
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, D) or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k/v must be [B, Hkv, N, D] with q's dtype")
    o = torch.empty_like(q) if o is None else o
    _cuda(q, o)
    with torch.cuda.device(dev):
        _check(lib().attn_causal_gqa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         B, Hq, Hkv, N, D, _dtype(q), _scale(scale), _stream(dev)),
               "attn_causal_gqa_fwd")
    return o


def causal_gqa_fwd_strided(q, k, v, o=None, scale=None):
    """Causal GQA prefill on strided views q [B,Hq,N,D], k/v [B,Hkv,N,D] (D
    contiguous), e.g. transposed projections or slices of a packed K/V tensor.
    o defaults to a new contiguous tensor."""
    dev = _cuda(q, k, v, strided=True)
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, D) or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k/v must be [B, Hkv, N, D] with q's dtype")
    o = torch.empty(q.shape, dtype=q.dtype, device=q.device) if o is None else o
    _cuda(q, o, strided=True)
    if o.shape != q.shape or o.dtype != q.dtype:
        raise ValueError("o must be [B, Hq, N, D] with q's dtype")
    with torch.cuda.device(dev):
        _check(lib().attn_causal_gqa_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                 o.data_ptr(), B, Hq, Hkv, N, D, _strides(q),
                                                 _strides(k), _strides(v), _strides(o), _dtype(q),
                                                 _scale(scale), _stream(dev)),
               "attn_causal_gqa_fwd_strided")
    return o


def rope_joint_workspace_bytes(B, H, N, D, dtype) -> int:
    return int(lib().attn_rope_joint_workspace_bytes(B, H, N, D, _dtype(torch.empty(0, dtype=dtype))))


def rope_joint_fwd(q, k, v, pos, axes_dim=(32, 32, 32, 32), theta=10000.0, o=None, scale=None,
                   workspace=None):
    """Multi-axis RoPE on q/k (positions pos [N,4] int32), then full attention."""
    dev = _cuda(q, k, v, pos)
    B, H, N, D = q.shape
    if k.shape != q.shape or v.shape != q.shape or pos.shape != (N, 4) or pos.dtype != torch.int32:
        raise ValueError("q/k/v [B,H,N,D] and pos int32 [N,4] required")
    o = torch.empty_like(q) if o is None else o
    need = rope_joint_workspace_bytes(B, H, N, D, q.dtype)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _cuda(q, o, workspace)
    with torch.cuda.device(dev):
        _check(lib().attn_rope_joint_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         B, H, N, D, pos.data_ptr(), _ints(axes_dim, 4),
                                         float(theta), _dtype(q), _scale(scale),
                                         workspace.data_ptr(), workspace.numel(), _stream(dev)),
               "attn_rope_joint_fwd")
    return o


def decode_workspace_bytes(B, Hq, Hkv, Lmax, D) -> int:
    return int(lib().attn_decode_gqa_workspace_bytes(B, Hq, Hkv, Lmax, D))


def decode_gqa(q, k_cache, v_cache, seq_len, o=None, scale=None, workspace=None, _ring=False):
    """GQA decode: q [B,Hq,D], caches [B,Hkv,Lmax,D], seq_len int32 [B] -> o [B,Hq,D].

    ``workspace`` (uint8, decode_workspace_bytes(...) bytes) must be zero-filled
    before its first use; calls leave it reusable.  If omitted a zeroed one is
    allocated for this call.
    """
    entry = "attn_decode_gqa_ring" if _ring else "attn_decode_gqa"
    dev = _cuda(q, k_cache, v_cache, seq_len)
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    if k_cache.shape != (B, Hkv, Lmax, D) or v_cache.shape != k_cache.shape or \
            seq_len.shape != (B,) or seq_len.dtype != torch.int32:
        raise ValueError("caches [B,Hkv,Lmax,D] and seq_len int32 [B] required")
    o = torch.empty_like(q) if o is None else o
    need = decode_workspace_bytes(B, Hq, Hkv, Lmax, D)
    if workspace is None:
        workspace = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    _cuda(q, o, workspace)
    with torch.cuda.device(dev):
        _check(getattr(lib(), entry)(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                     seq_len.data_ptr(), o.data_ptr(), B, Hq, Hkv, Lmax, D,
                                     _dtype(q), _scale(scale), workspace.data_ptr(),
                                     workspace.numel(), _stream(dev)),
               entry)
    return o


def decode_gqa_ring(q, k_cache, v_cache, seq_len, o=None, scale=None, workspace=None):
    """GQA decode over a ring cache: seq_len[b] counts every token appended
    (it may exceed Lmax); attends to the min(seq_len[b], Lmax) rows in use."""
    return decode_gqa(q, k_cache, v_cache, seq_len, o, scale, workspace, _ring=True)


def kv_append(k_cache, v_cache, k_new, v_new, seq_len, advance=True, _ring=False):
    """Write k_new/v_new [B,Hkv,D] into row seq_len[b] of the caches [B,Hkv,Lmax,D]
    (device-side position); with advance, seq_len[b] += 1 on the device."""
    entry = "attn_kv_append_ring" if _ring else "attn_kv_append"
    dev = _cuda(k_cache, v_cache, k_new, v_new, seq_len)
    B, Hkv, Lmax, D = k_cache.shape
    if v_cache.shape != k_cache.shape or k_new.shape != (B, Hkv, D) or v_new.shape != k_new.shape \
            or seq_len.shape != (B,) or seq_len.dtype != torch.int32:
        raise ValueError("caches [B,Hkv,Lmax,D], new rows [B,Hkv,D], seq_len int32 [B] required")
    with torch.cuda.device(dev):
        _check(getattr(lib(), entry)(k_cache.data_ptr(), v_cache.data_ptr(), k_new.data_ptr(),
                                     v_new.data_ptr(), seq_len.data_ptr(), B, Hkv, Lmax, D,
                                     _dtype(k_cache), 1 if advance else 0, _stream(dev)),
               entry)


def kv_append_ring(k_cache, v_cache, k_new, v_new, seq_len, advance=True):
    """Ring-cache append: row seq_len[b] % Lmax (the oldest token's row once
    the ring is full); with advance, seq_len[b] += 1 on the device."""
    kv_append(k_cache, v_cache, k_new, v_new, seq_len, advance, _ring=True)


def na3d_fwd(q, k, v, grid, kernel, o=None, scale=None):
    """3D neighborhood attention; q/k/v [B, heads, T*Hg*W, D]."""
    dev = _cuda(q, k, v)
    B, Hh, N, D = q.shape
    T, Hg, W = (int(x) for x in grid)
    if N != T * Hg * W or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q/k/v must be [B, heads, T*Hg*W, D]")
    o = torch.empty_like(q) if o is None else o
    _cuda(q, o)
    with torch.cuda.device(dev):
        _check(lib().attn_na3d_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   B, Hh, T, Hg, W, D, _ints(kernel, 3), _dtype(q),
                                   _scale(scale), _stream(dev)),
               "attn_na3d_fwd")
    return o


def na3d_fwd_strided(q, k, v, grid, kernel, o=None, scale=None):
    """3D neighborhood attention on strided [B, heads, T*Hg*W, D] views (D
    contiguous, tokens at a uniform stride), e.g. q.transpose(1, 2) of a
    [B, T*Hg*W, heads, D] projection. o defaults to a new contiguous tensor."""
    dev = _cuda(q, k, v, strided=True)
    B, Hh, N, D = q.shape
    T, Hg, W = (int(x) for x in grid)
    if N != T * Hg * W or k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype \
            or v.dtype != q.dtype:
        raise ValueError("q/k/v must be [B, heads, T*Hg*W, D] with one dtype")
    o = torch.empty(q.shape, dtype=q.dtype, device=q.device) if o is None else o
    _cuda(q, o, strided=True)
    if o.shape != q.shape or o.dtype != q.dtype:
        raise ValueError("o must be [B, heads, T*Hg*W, D] with q's dtype")
    with torch.cuda.device(dev):
        _check(lib().attn_na3d_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                           B, Hh, T, Hg, W, D, _ints(kernel, 3), _strides(q),
                                           _strides(k), _strides(v), _strides(o), _dtype(q),
                                           _scale(scale), _stream(dev)),
               "attn_na3d_fwd_strided")
    return o


def na3d_window_starts(grid, kernel, device=None):
    """int32 [T*Hg*W, 3] window starts from the kernels' own device function."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    T, Hg, W = (int(x) for x in grid)
    out = torch.empty((T * Hg * W, 3), dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(lib().attn_na3d_window_starts(T, Hg, W, _ints(kernel, 3), out.data_ptr(),
                                             _stream(dev)),
               "attn_na3d_window_starts")
    return out


def device_status(device=None) -> int:
    """Syncs the current stream and returns (and clears) the device error status."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib().attn_device_status(_stream(dev)))


def debug_wait_test(limit_ns: int, device=None) -> None:
    """One bounded device wait that is made to run out after limit_ns (testing
    the failure path): the next device_status() reports the timeout."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(lib().attn_debug_wait_test(int(limit_ns), _stream(dev)), "debug_wait_test")


def launch_count(family: str) -> int:
    return int(lib().attn_launch_count(FAMILIES[family]))


def version() -> str:
    return lib().attn_version().decode()
