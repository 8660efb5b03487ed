"""Host-side rules of the benchmark: a timed region whose clock record shows
a hardware or thermal slowdown, or SM clocks stuck far below their maximum
with no reason active, is invalid (it is taken again), while the power cap
alone is not; the clock record keeps the samples taken inside the timed
region; the sustained peak rates a region that lasts seconds or ran under
the power cap, the burst peak any other; and the per-step median and
minimum of a kernel's times."""

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


def _row(t, sm, reasons=(), mx="2070"):
    flags = ["Active" if r in reasons else "Not Active" for r in bench._CLOCK_REASONS]
    return [t, "0", str(sm), mx, "900.0", "0x0"] + flags


def test_clock_summary_keeps_the_timed_region():
    rows = [_row(10.0, 2070), _row(10.1, 2070), _row(10.6, 1500, ["sw_power_cap"]),
            _row(10.7, 1520, ["sw_power_cap"]), _row(11.5, 2070)]
    c = bench._summarise_clocks(rows, window=(10.55, 10.75))
    assert c["samples_in_timed_region"] == 2 and c["window"] == "timed region"
    assert c["sm_mhz"] == 1510.0 and c["reasons"] == ["sw_power_cap"]
    # a region shorter than the sampling interval: every sample counts
    c = bench._summarise_clocks(rows, window=(10.3, 10.31))
    assert c["samples_in_timed_region"] == 0 and c["samples"] == 5
    assert c["sm_mhz"] == 2070.0 and c["reasons"] == ["sw_power_cap"]
    # no window: every sample, and no window fields
    assert "window" not in bench._summarise_clocks(rows)


def test_nvsmi_timestamps_parse():
    t = bench._parse_nvsmi_time("2026/12/03 07:25:22.250")
    assert t is not None and abs(t % 1 - 0.25) < 1e-6
    assert bench._parse_nvsmi_time("n/a") is None


def test_peak_regime():
    capped = _c(["sw_power_cap"], sm=1777.0)
    # only a timed region of seconds is rated against the sustained figure
    assert bench._peak_regime(2500.0, _c([]), True, False)[0]
    assert bench._peak_regime(2500.0, capped, True, False)[0]
    # shorter regions (power-capped or not), graph replays and a missing
    # sustained figure are rated against the burst figure
    assert not bench._peak_regime(420.0, capped, True, False)[0]
    assert "sw_power_cap" in bench._peak_regime(420.0, capped, True, False)[1]
    assert not bench._peak_regime(8.0, _c([]), True, False)[0]
    assert not bench._peak_regime(8.0, _c(["sw_power_cap"], sm=2060.0), True, False)[0]
    assert not bench._peak_regime(2500.0, capped, True, True)[0]
    assert not bench._peak_regime(2500.0, capped, False, False)[0]


def test_alu_promotion_peak():
    """The block-scaled GEMM's CUDA-core ceiling: 64 GEMM FLOP per FP32 FMA,
    128 FMAs per SM per clock, every SM, the maximum SM clock."""
    class Props:
        multi_processor_count = 152

    class FakeTorch:
        class cuda:
            @staticmethod
            def get_device_properties(dev):
                return Props()

    peak, src = bench._alu_promotion_peak(FakeTorch, 0)
    assert abs(peak - 64 * 128 * 152 * 2070e6 / 1e12) < 1e-6    # 2578.4 TFLOP/s
    assert "128 FP32 FMA per SM per clock" in src and "152 SMs" in src


def test_per_op_splits_launches_in_step_order():
    W = {"per_op": [("a", 2e12), ("b", 4e12)]}
    phases = {"launches": {"gemm": [1.0, 2.0, 3.0, 2.0]}}   # steps: (a 1, b 2), (a 3, b 2)
    out = bench._per_op(W, phases, alu_peak=4000.0, fp8_peak=8000.0)
    assert abs(out["a"]["ms"] - 2.0) < 1e-12 and abs(out["b"]["ms"] - 2.0) < 1e-12
    assert abs(out["a"]["tflops"] - 1000.0) < 1e-9 and abs(out["b"]["tflops"] - 2000.0) < 1e-9
    assert abs(out["b"]["frac"] - 0.5) < 1e-12 and abs(out["b"]["frac_of_fp8_peak"] - 0.25) < 1e-12
    assert bench._per_op(W, {"launches": {"gemm": [1.0, 2.0, 3.0]}}, 1.0, 1.0) is None
