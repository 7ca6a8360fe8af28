"""The allocation-free decode entry point against the workspace one.

attn_decode_gqa_noalloc exists for callers that cannot give the library a
workspace (a host whose allocator owns all device memory and passes plugins
only tensors, or a decode loop that must not call cudaMalloc between tokens).
It keeps its split partials in a fixed array inside the library, so this test
calls it twice in a row through the C ABI -- the second call sees whatever the
first left in that array -- and checks both outputs against the fp64 oracle
and against attn_decode_gqa with a caller-owned workspace, within the bf16
tolerance of the parity tests.  The cases cover the decode workload, ragged
lengths, a single split per (batch, kv-head) and a problem whose partials fill
the array to within 1% of its 4 MiB.
The file sorts last so a failure here does not hide the other GPU tests.
"""
import ctypes

import numpy as np
import pytest

import oracle
from tests.util import assert_close, to_dev, to_host64
from workloads import WORKLOADS, make_inputs, to_f64

pytestmark = pytest.mark.gpu


def _noalloc(ta):
    L = ta.lib()
    fn = L.attn_decode_gqa_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_float, vp]
    fn.restype = i
    return fn


_NEAR_LIMIT_LENS = tuple(int(x) for x in np.random.default_rng(7902).integers(1, 65, size=125))


@pytest.mark.parametrize("name,overrides", [
    ("gqa_decode", {}),
    ("gqa_decode", dict(B=3, H=12, Hkv=4, D=64, Lmax=777, seq_len=(1, 777, 300), seed=7900)),
    # Lmax below 512 rows: one split per (batch, kv-head)
    ("gqa_decode", dict(B=2, H=8, Hkv=2, D=128, Lmax=200, seq_len=(200, 37), seed=7901)),
    # 1000 (batch, kv-head) pairs x 8 heads x 128 channels: 4,164,000 of 4,194,304 bytes
    ("gqa_decode", dict(B=125, H=64, Hkv=8, D=128, Lmax=64, seq_len=_NEAR_LIMIT_LENS, seed=7902)),
    # 8 (batch, kv-head) pairs of 4096 rows: 16 splits each, more than the
    # merge that requests every split at once takes (its general loop runs)
    ("gqa_decode", dict(B=1, H=32, Hkv=8, D=128, Lmax=4096, seq_len=(4096,), seed=7903)),
])
def test_noalloc_decode_matches_workspace_decode_twice(name, overrides):
    import torch
    from transformer_attention_tcgen05_gb300.build import build
    build()
    import transformer_attention_tcgen05_gb300 as ta
    torch.cuda.set_device(0)
    w = WORKLOADS[name].with_(**overrides)
    x = make_inputs(w)
    q, k, v = (to_dev(x[n], "bf16") for n in "qkv")
    sl = torch.from_numpy(x["seq_len"]).cuda()
    ref = to_host64(ta.decode_gqa(q, k, v, sl))        # workspace path
    exact = oracle.decode_gqa(to_f64(x["q"], "bf16"), to_f64(x["k"], "bf16"),
                              to_f64(x["v"], "bf16"), x["seq_len"])
    assert_close(ref, exact, "bf16", "workspace decode vs oracle")
    fn = _noalloc(ta)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    B, Hq, D = x["q"].shape
    _, Hkv, Lmax, _ = x["k"].shape
    for call in range(2):
        o = torch.full_like(q, float("nan"))
        st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), sl.data_ptr(), o.data_ptr(),
                B, Hq, Hkv, Lmax, D, 1, ctypes.c_float(0.0), stream)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert ta.device_status() == 0
        assert_close(to_host64(o), exact, "bf16", f"noalloc call {call} vs oracle")
        assert_close(to_host64(o), ref, "bf16", f"noalloc call {call} vs workspace decode")


def test_noalloc_rejects_problems_beyond_its_array():
    import torch
    import transformer_attention_tcgen05_gb300 as ta
    fn = _noalloc(ta)
    fake = ctypes.c_void_p(0x100000)      # never dereferenced: the size check comes first
    # 4096 (batch, kv-head) pairs with 8 padded heads of 128 channels cannot fit 4 MiB
    st = fn(fake, fake, fake, fake, ctypes.c_void_p(0x200000), 512, 64, 8, 64, 128, 1,
            ctypes.c_float(0.0), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 3      # ATTN_ERR_RESOURCE
