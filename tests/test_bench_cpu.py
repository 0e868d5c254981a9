"""bench.py host logic without a GPU: the clock-sample parser keeps the samples of the timed
region and reports every throttle reason seen there."""
import datetime
import os
import sys
import time

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402


def _line(t, mhz, power_cap="Not Active", thermal="Not Active"):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{ts}, 0, {mhz}, 2070, 900.5, 0x0, Not Active, Not Active, {thermal}, {power_cap}"


def test_clock_samples_restricted_to_timed_region():
    t0 = time.time()
    lines = [_line(t0 - 0.4, 1000), _line(t0 + 0.02, 2000), _line(t0 + 0.12, 1900, power_cap="Active"),
             _line(t0 + 0.6, 1500, thermal="Active"), "garbage"]
    c = bench.Clocks(0)
    c.lines, c.window = lines, (t0, t0 + 0.2)
    s = c.summary()
    assert s["samples"] == 2 and s["in_timed_region"]
    assert s["sm_mhz"] == 1950.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]          # the thermal sample lies outside the region


def test_clock_samples_fall_back_to_all_when_none_inside():
    t0 = time.time()
    c = bench.Clocks(0)
    c.lines, c.window = [_line(t0 - 1.0, 1200), _line(t0 + 2.0, 1800, thermal="Active")], (t0, t0 + 0.1)
    s = c.summary()
    assert s["samples"] == 2 and not s["in_timed_region"]
    assert s["reasons"] == ["sw_thermal_slowdown"]
