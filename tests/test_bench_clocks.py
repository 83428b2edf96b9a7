"""Which clock records void a timed region (bench.py re-measures it once):
thermal and hardware slowdowns, or an SM clock far below its maximum with no
reason given; the power cap alone is kept and noted."""
import bench


def test_power_cap_is_kept():
    assert bench.clocks_rejected({"sm_mhz": 1600.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}) is None
    assert bench.clocks_rejected({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}) is None


def test_slowdowns_are_rejected():
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        why = bench.clocks_rejected({"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap", r]})
        assert why is not None and r in why


def test_low_clock_without_reason_is_rejected():
    assert bench.clocks_rejected({"sm_mhz": 1200.0, "sm_max_mhz": 2070.0, "reasons": []}) is not None
    assert bench.clocks_rejected({"sm_mhz": 1200.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}) is None


def test_missing_samples_are_not_rejected():
    assert bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}) is None
