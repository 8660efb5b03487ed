"""Host-side rules of the benchmark: a timed region whose clock record shows
a hardware or thermal slowdown, or SM clocks stuck far below their maximum
with no reason active, is invalid (it is taken again), while the power cap
alone is not; and the per-step median and minimum of a kernel's times."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _c(reasons, sm=2070.0, mx=2070.0):
    return {"reasons": reasons, "sm_mhz": sm, "sm_max_mhz": mx, "samples": 10}


def test_slowdowns_invalidate():
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench._clocks_invalid(_c([r]))
        assert bench._clocks_invalid(_c(["sw_power_cap", r], sm=1500.0))


def test_power_cap_alone_is_valid():
    assert not bench._clocks_invalid(_c(["sw_power_cap"], sm=1260.0))


def test_low_clock_without_reason_is_a_lock():
    assert bench._clocks_invalid(_c([], sm=1000.0))
    assert not bench._clocks_invalid(_c([], sm=1900.0))


def test_no_samples_is_not_judged():
    assert not bench._clocks_invalid({"reasons": [], "sm_mhz": None, "sm_max_mhz": None,
                                      "samples": 0})


def test_median_min_per_step():
    xs = [1.0, 2.0, 3.0, 4.0, 5.0, 6.0]          # 3 steps x 2 launches
    assert bench._median_min_per_step(xs, 3) == [7.0, 3.0]
    assert bench._median_min_per_step([], 3) is None
    assert bench._median_min_per_step([1.0, 2.0], 3) is None
