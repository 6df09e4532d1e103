"""Host-side logic of bench.py that needs no GPU: the choice of the peak a timed region is
held to, and the clock-sample summary restricted to the samples inside the timed region."""
import bench


def _line(mhz, power, capped=False, thermal=False):
    act = lambda on: "Active" if on else "Not Active"  # noqa: E731
    return f"0, {mhz}, 2070, {power}, 0x0, Not Active, Not Active, {act(thermal)}, {act(capped)}"


def test_short_region_uses_burst_peak_long_region_sustained():
    peaks = {"bf16_tflops": 1885.7, "bf16_tflops_sustained": 1678.1}
    assert bench.region_peak_key(0.017, peaks) == "bf16_tflops"
    assert bench.region_peak_key(0.35, peaks) == "bf16_tflops"
    assert bench.region_peak_key(3.0, peaks) == "bf16_tflops_sustained"
    assert bench.region_peak_key(3.0, {"bf16_tflops": 1.0}) == "bf16_tflops"
    # a short region that the power controller already throttled is held to the sustained peak
    capped = {"sm_mhz": 1642.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    full = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.region_peak_key(0.36, peaks, capped) == "bf16_tflops_sustained"
    assert bench.region_peak_key(0.017, peaks, full) == "bf16_tflops"


def test_clock_summary_keeps_the_samples_inside_the_window():
    cs = bench.ClockSampler(0, interval_ms=20)
    cs.lines = [(0.0, _line(2070, 180)), (1.00, _line(1900, 1300, capped=True)),
                (1.02, _line(1850, 1350, capped=True)), (2.0, _line(2070, 200))]
    cs.proc = None
    inside = [x for x in cs.lines if 0.99 <= x[0] <= 1.05]
    out = bench.ClockSampler.summarise(inside)
    assert out["samples"] == 2 and out["sm_mhz"] == 1875.0 and out["reasons"] == ["sw_power_cap"]
    assert out["power_w"] == 1325.0
    every = bench.ClockSampler.summarise(cs.lines)
    assert every["samples"] == 4 and every["sm_max_mhz"] == 2070.0


def test_thermal_reason_is_reported():
    out = bench.ClockSampler.summarise([(0.0, _line(1500, 1000, thermal=True))])
    assert out["reasons"] == ["sw_thermal_slowdown"]


def test_nvml_summary_keeps_the_samples_inside_the_window():
    s = bench.NvmlClockSampler.__new__(bench.NvmlClockSampler)
    s.ok, s.interval_ms, s.max_mhz = True, 1.0, 2070.0
    s._stop = bench.threading.Event()
    s.t = bench.threading.Thread(target=lambda: None)
    s.t.start()
    s.samples = [(0.0, 2070.0, 2070.0, 180.0, 0), (1.001, 1900.0, 2070.0, 1300.0, 0x4),
                 (1.002, 1800.0, 2070.0, 1350.0, 0x4 | 0x20), (2.0, 2070.0, 2070.0, 200.0, 0)]
    out = s.stop(window=(1.0, 1.01))
    assert out["samples"] == 2 and out["sm_mhz"] == 1850.0 and out["in_region"]
    assert out["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]
    assert out["source"] == "nvml"
