"""bench.py's summary of the clock samples taken during the timed region (nvidia-smi lines in
the order index, clocks.sm, clocks.max.sm, power.draw, reasons.active, hw_slowdown,
hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap)."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_median_max_and_active_reasons():
    text = "\n".join([
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1200.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    ])
    r = bench.parse_clock_samples(text)
    assert r == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_thermal_and_hw_reasons_are_reported():
    text = ("0, 1500, 2070, 1000, 0x48, Active, Active, Not Active, Not Active\n"
            "0, 1600, 2070, 1000, 0x20, Not Active, Not Active, Active, Not Active\n")
    r = bench.parse_clock_samples(text)
    assert r["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert r["sm_mhz"] == 1550.0


def test_unparseable_lines_are_skipped():
    text = ("garbage\n"
            "0, [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]\n"
            "0, 2070, 2070, 800, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    r = bench.parse_clock_samples(text)
    assert r["samples"] == 1 and r["reasons"] == []


def test_no_samples():
    assert bench.parse_clock_samples("") == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                                             "samples": 0}
