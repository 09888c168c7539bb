"""Host-side logic of bench.py that needs no GPU: the clock record kept
beside each measurement."""
import datetime
import time

import bench


def _line(t, sm, power_cap="Not Active", hw="Not Active"):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return (f"{ts}, 0, {sm}, 2070, 1200.5, 0x0000000000000000, {hw}, Not Active, Not Active, "
            f"{power_cap}")


def test_clocks_keep_only_the_timed_window():
    t = time.time()
    lines = [_line(t - 0.3, 1200), _line(t + 0.01, 2070), _line(t + 0.06, 2055, power_cap="Active"),
             _line(t + 0.5, 900, hw="Active")]
    c = bench.Clocks.parse(lines, (t, t + 0.1))
    assert c["in_timed_region"] and c["samples"] == 2
    assert c["sm_mhz"] in (2055.0, 2070.0) and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]  # the hw_slowdown outside the window is not counted


def test_clocks_fall_back_to_every_sample_when_none_is_inside():
    t = time.time()
    lines = [_line(t - 1.0, 2070), _line(t - 0.9, 2070, hw="Active")]
    c = bench.Clocks.parse(lines, (t, t + 0.1))
    assert not c["in_timed_region"] and c["samples"] == 2
    assert c["reasons"] == ["hw_slowdown"]


def test_clocks_ignore_malformed_lines():
    c = bench.Clocks.parse(["", "not, a, sample", "[N/A]"], None)
    assert c["samples"] == 0 and c["sm_mhz"] is None
