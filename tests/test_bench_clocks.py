"""The benchmark's reading of nvidia-smi clock samples, on CPU: the median SM clock is
taken over the samples under load (the idle lead-in is left out) and every throttle
reason seen in any sample is reported."""
import bench


def _line(sm, smax, watts, sw_cap="Not Active", hw="Not Active"):
    # index, clocks.sm, clocks.max.sm, power.draw, reasons.active, hw_slowdown,
    # hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    return f"0, {sm}, {smax}, {watts}, 0x0, {hw}, Not Active, Not Active, {sw_cap}"


def test_median_over_load_samples_only():
    lines = [_line(2070, 2070, 180.0), _line(2070, 2070, 190.0),            # idle lead-in
             _line(1550, 2070, 720.0, sw_cap="Active"), _line(1620, 2070, 700.0),
             _line(1740, 2070, 650.0)]
    c = bench.parse_clock_samples("\n".join(lines))
    assert c["samples"] == 5 and c["load_samples"] == 3
    assert c["sm_mhz"] == 1620.0           # median of 1550, 1620, 1740; idle 2070s excluded
    assert c["sm_max_mhz"] == 2070.0
    assert c["power_w_max"] == 720.0
    assert c["reasons"] == ["sw_power_cap"]


def test_unavailable_power_keeps_every_sample():
    lines = [_line(2070, 2070, "[N/A]"), _line(1900, 2070, "[N/A]"),
             _line(1800, 2070, "[N/A]", hw="Active")]
    c = bench.parse_clock_samples("\n".join(lines))
    assert c["power_w_max"] is None and c["load_samples"] == 3
    assert c["sm_mhz"] == 1900.0
    assert c["reasons"] == ["hw_slowdown"]


def test_no_samples():
    assert bench.parse_clock_samples("") is None
    assert bench.parse_clock_samples("garbage line\n") is None
