"""bench.py's host logic on CPU (no GPU).

* The clock and throttle summary of the timed window.
* The roofline of a shape and the algorithmic figures the JSON line reports.  They are checked against
  the roofline table worked out from the method's stated costs, with a 6776.3 GB/s copy and a
  1912.5 TFLOP/s bf16 rate: 39.8 us forward and 79.2 us backward at B = 4, H = 16, N = 4096, D = 128,
  every call HBM-bound.
  * Forward: Q, K, V read, O and the fp32 normaliser written; 4 D^2 flops per row.
  * Backward: eight tensor volumes; 10 D^2 flops per row.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_standard_shape_roofline():
    fwd, bwd = bench.shape_roofline_s(4, 16, 4096, 128, 6776.3, 1912.5)
    assert fwd * 1e6 == pytest.approx(39.8, abs=0.05)
    assert bwd * 1e6 == pytest.approx(79.2, abs=0.05)
    # the bench line's own figures for that shape agree with the sweep's helper
    assert bench.alg_bytes("fwd") == 4 * 4 * 16 * 4096 * 128 * 2 + 4 * 4 * 16 * 4096
    assert bench.alg_bytes("bwd") == 8 * 4 * 16 * 4096 * 128 * 2
    assert bench.alg_bytes("fwd") / (6776.3e9) == pytest.approx(fwd)


@pytest.mark.parametrize("D,fwd_us,bwd_us", [(32, 10.1, 19.8), (64, 20.0, 39.6), (256, 79.4, 158.5)])
def test_head_size_rooflines(D, fwd_us, bwd_us):
    fwd, bwd = bench.shape_roofline_s(4, 16, 4096, D, 6776.3, 1912.5)
    assert fwd * 1e6 == pytest.approx(fwd_us, abs=0.1)
    assert bwd * 1e6 == pytest.approx(bwd_us, abs=0.1)


def test_intensity_stays_below_the_ridge():
    """Flops per byte of every call of the sweep stay below the ridge (1912.5 TF / 6776.3 GB/s = 282):
    the roofline of each is its bytes."""
    for _, b, h, n, d, _, _ in bench.SWEEP_CASES:
        t = b * h * n * d * 2
        assert 4 * d * d * b * h * n / (4 * t + 4 * b * h * n) < 282
        assert 10 * d * d * b * h * n / (8 * t) < 282


def test_sweep_cases_are_the_measured_workloads():
    names = [c[0] for c in bench.SWEEP_CASES]
    assert names == ["head_size_D32", "head_size_D64", "head_size_D256", "seq_len_N1024", "seq_len_N2048",
                     "seq_len_N8192", "seq_len_N16384", "seq_len_N32768", "seq_len_N65536", "decoder_24_layers"]
    assert bench.SWEEP_CASES[-1][1:] == (8, 16, 2048, 128, 24, 4)


def _row(sm, mx, pw, active, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return ["0", str(sm), str(mx), str(pw), active, hw, hwt, swt, cap]


def test_clock_summary_takes_the_window_median_and_active_reasons():
    s = bench.ClockSampler(0)
    s.samples = [(0.5, _row(1200, 2070, 300, "0x0")),            # before the window: ignored
                 (1.0, _row(2070, 2070, 700, "0x0")),
                 (1.2, _row(2040, 2070, 720, "0x4", cap="Active")),
                 (1.4, _row(2070, 2070, 710, "0x0")),
                 (9.0, _row(120, 2070, 90, "0x0", hwt="Active"))]  # after the window: ignored
    out = bench.ClockSampler.summary(s, 1.0, 2.0)
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_w_max"] == 720


def test_clock_summary_reports_thermal_and_hardware_slowdowns():
    s = bench.ClockSampler(0)
    s.samples = [(1.0, _row(1500, 2070, 900, "0x40", hw="Active")),
                 (1.1, _row(1400, 2070, 900, "0x20", swt="Active")),
                 (1.2, _row("[N/A]", 2070, "[N/A]", "0x0", hwt="Active"))]
    out = bench.ClockSampler.summary(s, 0.0, 2.0)
    assert out["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert out["sm_mhz"] == 1450  # unreadable samples are skipped
    assert bench.ClockSampler.summary(bench.ClockSampler(0), 0.0, 1.0)["samples"] == 0


@pytest.mark.parametrize("args", [["--batch", "8"], ["--head-dim", "64"], ["--layout", "bnhd"]])
def test_other_shapes_time_the_hot_path_only(args):
    """The bench line is the standard workload: another batch, head size or layout is refused unless
    --profile (the hot path alone, for profilers) is given; the refusal comes before any GPU work."""
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args, "--steps", "1"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 2
    assert "--profile" in r.stderr
