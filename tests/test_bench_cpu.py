"""Host-side pieces of bench.py that need no GPU: the full-row parity summary
and the clock sampler's behaviour when no GPU telemetry is available."""
import numpy as np


def test_parity_summary_metrics_and_bounds():
    import bench
    ref = np.random.default_rng(0).standard_normal((3, 5, 64))
    got = ref.copy()
    got[0, 0, 0] += 1e-2                      # one element off by 1e-2
    e = bench.parity_of(got, ref)
    assert e["rows"] == 15
    assert abs(e["max_abs"] - 1e-2) < 1e-12
    assert abs(e["mean_abs"] - 1e-2 / got.size) < 1e-15
    assert e["within_tol"]
    got[1, 2, 3] += 0.5                       # beyond the 2e-2 max-abs bound
    assert not bench.parity_of(got, ref)["within_tol"]
    got = ref.copy()
    got[2, 4, 5] = np.nan
    assert not bench.parity_of(got, ref)["within_tol"]


def test_clock_sampler_without_telemetry_reports_nothing():
    import bench
    cs = bench.ClockSampler(0)
    cs.nvml = None
    cs.start()
    out = cs.stop()
    assert out is None or set(out) >= {"sm_mhz", "sm_max_mhz", "samples", "reasons"}
