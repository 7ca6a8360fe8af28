"""Failure reporting on the GPU without a fault: a bounded wait that runs out.

Every spin-wait of the attention kernels (mbarrier phases, TMA completion,
tensor-core commits) gives up after a limit, raises the device error word and
lets its CTA return.  attn_debug_wait_test launches one such wait on a barrier
that nothing ever completes, with a short limit; the host must then read
ATTN_ERR_TIMEOUT, the read must clear it, and the context must still run the
attention kernels correctly afterwards.
"""
import numpy as np
import pytest

import oracle
from tests.util import assert_close, to_dev, to_host64
from workloads import WORKLOADS, make_inputs, to_f64

pytestmark = pytest.mark.gpu

ATTN_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def ta():
    import torch
    from transformer_attention_tcgen05_gb300.build import build
    build()
    import transformer_attention_tcgen05_gb300 as ta
    torch.cuda.set_device(0)
    return ta


@pytest.mark.parametrize("limit_ns", [1_000, 2_000_000])
def test_bounded_wait_runs_out_and_reports_timeout(ta, limit_ns):
    import time
    assert ta.device_status() == 0
    n0 = ta.launch_count("debug")
    t0 = time.perf_counter()
    ta.debug_wait_test(limit_ns)
    st = ta.device_status()                  # synchronises: the wait has returned
    elapsed = time.perf_counter() - t0
    assert ta.launch_count("debug") == n0 + 1
    assert st == ATTN_ERR_TIMEOUT
    assert ta.device_status() == 0           # the read cleared the word
    assert elapsed < 5.0                     # bounded: far below any hang
    # the context is still usable: a tensor-core call right after is correct
    w = WORKLOADS["na3d_21x60x104_k11"].with_(grid=(4, 12, 20), kernel=(3, 5, 7), H=1,
                                             N=4 * 12 * 20, seed=8950)
    x = make_inputs(w)
    n1 = ta.launch_count("tc_na")
    o = ta.na3d_fwd(*(to_dev(x[n], "bf16") for n in "qkv"), w.grid, w.kernel)
    assert ta.launch_count("tc_na") > n1
    ref = oracle.na3d_fwd(*(to_f64(x[n], "bf16") for n in "qkv"), w.grid, w.kernel)
    assert_close(to_host64(o), ref, "bf16", "after a timeout")
    assert ta.device_status() == 0
