"""Host logic of bench.py that needs no GPU: the clock summary that rejects a
throttled or clock-locked run reads the sampled SM clocks and clock-event
reason bits correctly, and the sampler degrades to no samples (not an error)
where no GPU management library is present."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_clock_summary_median_max_and_reasons():
    cs = bench.ClockSampler(0)
    # (SM MHz, max SM MHz, NVML clock-event reason bits)
    cs.samples = [(1900.0, 2070.0, 0x0), (2000.0, 2070.0, 0x4), (2070.0, 2070.0, 0x1), (1800.0, 2070.0, 0x8)]
    s = cs.summary()
    assert s["sm_mhz"] == 1950.0
    assert s["sm_max_mhz"] == 2070.0
    # gpu_idle is never reported; power cap and hardware slowdown are
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert s["samples"] == 4


def test_clock_summary_without_samples():
    s = bench.ClockSampler(0).summary()
    assert s["sm_mhz"] is None and s["sm_max_mhz"] is None and s["samples"] == 0 and s["reasons"] == []


def test_sampler_context_is_safe_without_gpu():
    with bench.ClockSampler(0) as cs:
        pass
    s = cs.summary()
    assert s["samples"] >= 0 and isinstance(s["reasons"], list)


def test_reference_arm_sample_keeps_the_run_bounded():
    """The reference arm samples fewer weight rows a step when warmup + steps
    full oracle steps would run past its budget: the driver's short run keeps
    every row, a 20,000-step run a 32-row-aligned slice."""
    assert bench.reference_rows(7168, 0.9, 20, 5) == 7168
    rows = bench.reference_rows(7168, 0.9, 20000, 200)
    assert rows % 32 == 0 and 32 <= rows < 7168
    assert (20000 + 200) * 0.9 * rows / 7168 <= 150.0 + 0.9 * 32 / 7168 * 20200
    assert bench.reference_rows(7168, 100.0, 1000, 3) == 32
