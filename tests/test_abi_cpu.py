"""CPU checks of the C ABI: the library loads, exports every declared symbol,
and host-side validation rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from transformer_attention_tcgen05_gb300.build import build
    build()
    import transformer_attention_tcgen05_gb300 as ta
    return ta.lib()


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert "attn_full_fwd" in names and "attn_decode_gqa" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_no_undeclared_exports(L):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", L._name], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    ours = {n for n in exported if n.startswith("attn_")}
    assert ours == set(_declared()), ours ^ set(_declared())


def test_status_strings_and_version(L):
    L.attn_status_string.restype = ctypes.c_char_p
    assert L.attn_status_string(0) == b"ok"
    assert b"invalid" in L.attn_status_string(1)
    L.attn_version.restype = ctypes.c_char_p
    assert b"sm_103a" in L.attn_version()


def test_workspace_queries_are_host_arithmetic(L):
    import transformer_attention_tcgen05_gb300 as ta
    b = ta.decode_workspace_bytes(8, 32, 8, 4096, 128)
    assert b > 0 and b % 256 == 0
    assert ta.decode_workspace_bytes(8, 30, 8, 4096, 128) == 0       # Hq % Hkv != 0
    assert ta.decode_workspace_bytes(1, 32, 2, 4096, 128) == 0       # group of 16 unsupported
    import torch
    r = ta.rope_joint_workspace_bytes(1, 24, 4608, 128, torch.bfloat16)
    assert r >= 2 * 24 * 4608 * 128 * 2 and r % 256 == 0


FAKE = ctypes.c_void_p(0x10000)   # aligned, never dereferenced: validation fails first


def _full(L, *, q=FAKE, o=ctypes.c_void_p(0x20000), B=1, H=1, Nq=8, Nkv=8, D=32, dt=0):
    L.attn_full_fwd.restype = ctypes.c_int
    return L.attn_full_fwd(q, FAKE, FAKE, o, B, H, Nq, Nkv, D, dt, ctypes.c_float(0.0), None)


def test_full_validation(L):
    assert _full(L, q=None) == 1
    assert _full(L, q=ctypes.c_void_p(0x10004)) == 1      # misaligned
    assert _full(L, D=48) == 1
    assert _full(L, Nq=0) == 1
    assert _full(L, dt=7) == 1
    assert _full(L, dt=3) == 1                           # only F32 / BF16 / F16
    assert _full(L, dt=2, D=48) == 1                     # F16 is validated like the others
    assert _full(L, o=FAKE) == 1                         # output aliases an input


def _strided(L, qs, os_, *, B=2, H=3, N=16, D=64, dt=1):
    L.attn_full_fwd_strided.restype = ctypes.c_int
    S = ctypes.c_int64 * 3
    dense = S(H * N * D, N * D, D)
    return L.attn_full_fwd_strided(FAKE, FAKE, FAKE, ctypes.c_void_p(0x20000), B, H, N, N, D,
                                   S(*qs), dense, dense, S(*os_), dt, ctypes.c_float(0.0), None)


def test_full_strided_validation(L):
    """Only layouts that must be refused are passed: the pointers are fake."""
    H, N, D = 3, 16, 64
    dense = (H * N * D, N * D, D)
    assert _strided(L, (H * N * D, N * D, D + 4), dense) == 1    # row stride 136 bytes in bf16
    assert _strided(L, (H * N * D, 0, D), dense) == 1            # zero stride on an extent-3 axis
    assert _strided(L, (-H * N * D, N * D, D), dense) == 1       # negative stride
    assert _strided(L, dense, (H * N * D, N * D, D // 2)) == 1   # output rows overlap
    assert _strided(L, dense, (H * N * D, D, D)) == 1            # two heads share output rows
    assert _strided(L, dense, (N * D, N * D, D)) == 1            # batches share output heads
    assert _strided(L, (H * N * D, N * D, 6), dense, dt=0) == 1  # fp32 row stride 24 bytes
    L.attn_full_fwd_strided.restype = ctypes.c_int
    S = ctypes.c_int64 * 3
    assert L.attn_full_fwd_strided(FAKE, FAKE, FAKE, ctypes.c_void_p(0x20000), 1, 1, 8, 8, 64,
                                   None, S(512, 512, 64), S(512, 512, 64), S(512, 512, 64), 1,
                                   ctypes.c_float(0.0), None) == 1


def test_causal_strided_validation(L):
    """Only layouts that must be refused are passed: the pointers are fake."""
    L.attn_causal_gqa_fwd_strided.restype = ctypes.c_int
    S = ctypes.c_int64 * 3
    B, Hq, Hkv, N, D = 2, 4, 2, 16, 64
    q = S(Hq * N * D, N * D, D)
    kv = S(Hkv * N * D, N * D, D)

    def call(qs=q, ks=kv, os_=q, hq=Hq, hkv=Hkv):
        return L.attn_causal_gqa_fwd_strided(FAKE, FAKE, FAKE, ctypes.c_void_p(0x20000), B, hq,
                                             hkv, N, D, qs, ks, kv, os_, 1, ctypes.c_float(0.0),
                                             None)
    assert call(hq=3, hkv=2) == 1                                # Hq not a multiple of Hkv
    assert call(ks=S(Hkv * N * D, N * D, D + 2)) == 1            # K row stride 132 bytes
    assert call(os_=S(Hq * N * D, D, D)) == 1                    # heads share output rows
    assert call(qs=None) == 1


def test_na3d_strided_validation(L):
    """Only layouts that must be refused are passed: the pointers are fake."""
    L.attn_na3d_fwd_strided.restype = ctypes.c_int
    S = ctypes.c_int64 * 3
    B, H, T, Hg, W, D = 1, 2, 2, 4, 4, 64
    N = T * Hg * W
    ok = S(H * N * D, N * D, D)
    kern = (ctypes.c_int * 3)(3, 3, 3)

    def call(qs=ok, os_=ok, k=kern):
        return L.attn_na3d_fwd_strided(FAKE, FAKE, FAKE, ctypes.c_void_p(0x20000), B, H, T, Hg, W,
                                       D, k, qs, ok, ok, os_, 1, ctypes.c_float(0.0), None)
    assert call(qs=S(H * N * D, N * D, D + 4)) == 1              # token stride 136 bytes
    assert call(os_=S(H * N * D, D, H * D // 2)) == 1            # output tokens overlap
    assert call(k=(ctypes.c_int * 3)(3, 4, 3)) == 1              # even window


def test_na3d_validation(L):
    L.attn_na3d_fwd.restype = ctypes.c_int
    o = ctypes.c_void_p(0x20000)
    for kern in ([3, 4, 3], [0, 3, 3], [-1, 3, 3]):       # even / zero / negative
        k = (ctypes.c_int * 3)(*kern)
        assert L.attn_na3d_fwd(FAKE, FAKE, FAKE, o, 1, 1, 2, 4, 4, 32, k, 0,
                               ctypes.c_float(0.0), None) == 1
    k = (ctypes.c_int * 3)(3, 3, 3)
    assert L.attn_na3d_fwd(FAKE, FAKE, FAKE, o, 1, 1, 0, 4, 4, 32, k, 0,
                           ctypes.c_float(0.0), None) == 1


def test_decode_validation(L):
    L.attn_decode_gqa.restype = ctypes.c_int
    o = ctypes.c_void_p(0x20000)
    ws = ctypes.c_void_p(0x40000)
    f = ctypes.c_float(0.0)
    # Hq % Hkv != 0
    assert L.attn_decode_gqa(FAKE, FAKE, FAKE, FAKE, o, 1, 6, 4, 64, 128, 1, f, ws, 1 << 20, None) == 1
    # fp32 decode is not built (16-bit caches only)
    assert L.attn_decode_gqa(FAKE, FAKE, FAKE, FAKE, o, 1, 8, 2, 64, 128, 0, f, ws, 1 << 20, None) == 2
    # workspace too small (bf16 and f16 caches alike)
    assert L.attn_decode_gqa(FAKE, FAKE, FAKE, FAKE, o, 1, 8, 2, 64, 128, 1, f, ws, 16, None) == 3
    assert L.attn_decode_gqa(FAKE, FAKE, FAKE, FAKE, o, 1, 8, 2, 64, 128, 2, f, ws, 16, None) == 3
    # misaligned workspace
    assert L.attn_decode_gqa(FAKE, FAKE, FAKE, FAKE, o, 1, 8, 2, 64, 128, 1, f,
                             ctypes.c_void_p(0x40010), 1 << 20, None) == 1


def test_ring_entries_validate_like_their_linear_forms(L):
    """The ring decode and append entries share the linear ones' host checks
    (only refusals are passed: the pointers are fake)."""
    L.attn_decode_gqa_ring.restype = ctypes.c_int
    L.attn_kv_append_ring.restype = ctypes.c_int
    o = ctypes.c_void_p(0x20000)
    ws = ctypes.c_void_p(0x40000)
    f = ctypes.c_float(0.0)
    assert L.attn_decode_gqa_ring(FAKE, FAKE, FAKE, FAKE, o, 1, 6, 4, 64, 128, 1, f, ws, 1 << 20,
                                  None) == 1                      # Hq % Hkv != 0
    assert L.attn_decode_gqa_ring(FAKE, FAKE, FAKE, FAKE, o, 1, 8, 2, 64, 128, 0, f, ws, 1 << 20,
                                  None) == 2                      # fp32 cache
    assert L.attn_decode_gqa_ring(FAKE, FAKE, FAKE, FAKE, o, 1, 8, 2, 64, 128, 1, f, ws, 16,
                                  None) == 3                      # workspace too small
    assert L.attn_decode_gqa_ring(FAKE, FAKE, FAKE, None, o, 1, 8, 2, 64, 128, 1, f, ws, 1 << 20,
                                  None) == 1                      # no seq_len
    kc, vc = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x30000)
    new = ctypes.c_void_p(0x50000)
    assert L.attn_kv_append_ring(kc, kc, new, new, FAKE, 1, 2, 64, 64, 1, 1, None) == 1  # k is v
    assert L.attn_kv_append_ring(kc, vc, new, new, FAKE, 1, 2, 64, 48, 1, 1, None) == 1  # D = 48
    assert L.attn_kv_append_ring(kc, vc, new, new, None, 1, 2, 64, 64, 1, 1, None) == 1  # no seq_len


def test_rope_validation(L):
    L.attn_rope_joint_fwd.restype = ctypes.c_int
    o = ctypes.c_void_p(0x20000)
    ws = ctypes.c_void_p(0x40000)
    f = ctypes.c_float(0.0)
    bad = [(32, 32, 32, 30), (33, 31, 32, 32), (32, 32, 32, 33)]
    for ax in bad:
        a = (ctypes.c_int * 4)(*ax)
        assert L.attn_rope_joint_fwd(FAKE, FAKE, FAKE, o, 1, 2, 16, 128, FAKE, a,
                                     ctypes.c_float(1e4), 1, f, ws, 1 << 20, None) == 1
    a = (ctypes.c_int * 4)(32, 32, 32, 32)
    assert L.attn_rope_joint_fwd(FAKE, FAKE, FAKE, o, 1, 2, 16, 128, FAKE, a,
                                 ctypes.c_float(-1.0), 1, f, ws, 1 << 20, None) == 1   # theta
    assert L.attn_rope_joint_fwd(FAKE, FAKE, FAKE, o, 1, 2, 16, 128, FAKE, a,
                                 ctypes.c_float(1e4), 1, f, ws, 64, None) == 3         # workspace


def test_wait_test_limit_range_checked_on_the_host(L):
    L.attn_debug_wait_test.argtypes = [ctypes.c_uint64, ctypes.c_void_p]
    L.attn_debug_wait_test.restype = ctypes.c_int
    assert L.attn_debug_wait_test(999, None) == 1              # below 1 us
    assert L.attn_debug_wait_test(1_000_000_001, None) == 1    # above the 1 s wait limit


def test_launch_counter_unknown_family(L):
    L.attn_launch_count.restype = ctypes.c_uint64
    assert L.attn_launch_count(99) == 0
    assert L.attn_launch_count(-1) == 0


def test_product_path_does_not_import_oracle():
    import subprocess
    import sys
    code = ("import sys, transformer_attention_tcgen05_gb300 as ta; "
            "assert not any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules), 'oracle imported'")
    subprocess.run([sys.executable, "-c", code], cwd=ROOT, check=True)
    for fn in os.listdir(os.path.join(ROOT, "transformer_attention_tcgen05_gb300")):
        if fn.endswith(".py"):
            src = open(os.path.join(ROOT, "transformer_attention_tcgen05_gb300", fn)).read()
            assert "import oracle" not in src and "from oracle" not in src, fn
