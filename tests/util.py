"""Helpers shared by the GPU parity tests: host <-> device moves and error metrics."""
from __future__ import annotations

import numpy as np

from workloads import bf16_to_f32

# Tolerances: fp32 from the fp32 workload statement (max-abs 1e-4), bf16 from
# the bf16 statement (max-abs 2e-2, mean-abs 2e-3 with fp32 accumulation).
# The relative-RMS bounds are stricter additions: with N(0,1) inputs |O| is
# small (RMS ~ sqrt(e / window)), so the absolute bounds alone are ~1 sigma of
# O; a relative-RMS bound of 1e-2 (bf16) / 1e-5 (fp32) catches real bugs.
# f16 keeps 3 more mantissa bits than bf16 (P and O are rounded with relative
# error 2^-11 instead of 2^-8), so its bounds are the bf16 ones divided by 4,
# leaving a factor of two for accumulation order.
TOL = {
    "f32": dict(max_abs=1e-4, mean_abs=1e-5, rel_rms=1e-5),
    "bf16": dict(max_abs=2e-2, mean_abs=2e-3, rel_rms=1e-2),
    "f16": dict(max_abs=5e-3, mean_abs=5e-4, rel_rms=2.5e-3),
}


def to_dev(x: np.ndarray, dtype: str, device="cuda"):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def to_host64(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return bf16_to_f32(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    return t.detach().cpu().numpy().astype(np.float64)


def errors(got: np.ndarray, ref: np.ndarray) -> dict:
    d = np.abs(got - ref)
    return dict(max_abs=float(d.max()), mean_abs=float(d.mean()),
                rel_rms=float(np.sqrt(np.mean(d ** 2)) / max(np.sqrt(np.mean(ref ** 2)), 1e-30)),
                finite=bool(np.all(np.isfinite(got))))


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    e = errors(got, ref)
    tol = TOL[dtype]
    assert e["finite"], f"{what}: non-finite output"
    for k, lim in tol.items():
        assert e[k] <= lim, f"{what}: {k} {e[k]:.3e} > {lim:.1e} ({e})"
    return e
