"""The bench's clock record on CPU: nvidia-smi lines are parsed, only the
samples inside the busy window around the timed steps are kept, throttle
reasons are collected, and the busy window is sized from the step time."""
import datetime

import bench


def _line(t: float, sm: int, reasons=("Not Active",) * 4, watts="812.5") -> str:
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([stamp, str(sm), "2070", watts, "0x0000000000000000", *reasons])


def test_only_samples_inside_the_busy_window_count():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 0.25, 1200), _line(t0 - 0.05, 1200),            # idle, before the window
             _line(t0 + 0.1, 2040), _line(t0 + 0.2, 2010), _line(t0 + 0.3, 1995),
             _line(t0 + 1.4, 900)]                                        # after the window
    rec = bench.ClockSampler.summarize(lines, (t0, t0 + 1.0))
    assert rec["samples"] == 3
    assert rec["sm_mhz"] == 2010.0
    assert rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == []
    assert rec["power_w"] == 812.5
    assert rec["scope"].startswith("samples taken while")


def test_throttle_reasons_are_collected_by_name():
    t0 = 1_800_000_000.0
    lines = [_line(t0 + 0.1, 1900, ("Not Active", "Not Active", "Not Active", "Active")),
             _line(t0 + 0.2, 1700, ("Active", "Not Active", "Not Active", "Not Active")),
             _line(t0 + 0.3, 2070, watts="[N/A]")]
    rec = bench.ClockSampler.summarize(lines, (t0, t0 + 1.0))
    assert rec["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert rec["sm_mhz"] == 1900.0
    assert rec["power_w"] == 812.5


def test_no_sample_in_the_window_falls_back_to_all_and_says_so():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 1.0, 2070), "garbage line", _line(t0 + 5.0, 2050)]
    rec = bench.ClockSampler.summarize(lines, (t0, t0 + 0.001))
    assert rec["samples"] == 2
    assert rec["scope"].startswith("no sample fell inside")
    assert bench.ClockSampler.summarize(["", "a,b"], None) is None


def test_busy_window_is_sized_from_the_step_time():
    assert bench.busy_pad_steps(0.22) == round(bench.BUSY_PAD_S * 1e3 / 0.22)
    assert bench.busy_pad_steps(9.25) == round(bench.BUSY_PAD_S * 1e3 / 9.25)
    assert bench.busy_pad_steps(1e-6) == 20000
    assert bench.busy_pad_steps(1e4) == 1
    assert bench.busy_pad_steps(0.0) == 1
    assert bench.busy_pad_steps(float("nan")) == 1
