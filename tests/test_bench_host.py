"""Host-side logic of bench.py that needs no GPU: the clock-sample summary."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _line(sm, smax=2070, power=900.0, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return "%s, %s, %s, %s, %s, %s, %s" % (sm, smax, power, hw, hwt, swt, cap)


def test_samples_inside_the_timed_region_decide():
    lines = [(0.0, _line(600)), (0.1, _line(610)),                      # idle, before the region
             (1.0, _line(2070)), (1.1, _line(2055)), (1.2, _line(2070, cap="Active")),
             (2.5, _line(700, hwt="Active"))]                            # after the region
    c = bench.summarize_clocks(lines, region=(0.95, 1.18))
    assert c["samples_in_region"] == 3 and c["samples"] == 3
    assert c["sm_mhz"] == 2070 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]      # the sample read within 25 ms after the region counts


def test_a_region_shorter_than_the_sampling_period_falls_back_to_all_samples():
    lines = [(0.0, _line(2000)), (0.1, _line(2070)), (0.2, _line(1990, hw="Active"))]
    c = bench.summarize_clocks(lines, region=(0.31, 0.32))
    assert c["samples_in_region"] == 0 and c["samples"] == 3
    assert c["sm_mhz"] == 2000 and c["reasons"] == ["hw_slowdown"]


def test_malformed_lines_are_skipped():
    lines = [(0.0, "garbage"), (0.1, "[N/A], 2070, 1.0, a, b, c, d"), (0.2, _line(1980))]
    c = bench.summarize_clocks(lines)
    assert c["samples"] == 1 and c["sm_mhz"] == 1980
    assert bench.summarize_clocks([])["sm_mhz"] is None

