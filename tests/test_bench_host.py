"""Host logic of bench.py that needs no GPU: the clock-sample window."""
import datetime
import importlib.util
import os
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _stamp(t):
    return datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]


def _line(t, mhz, cap):
    act = "Active" if cap else "Not Active"
    return f"{_stamp(t)}, 0, {mhz}, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, {act}"


def test_clock_samples_outside_the_region_are_dropped():
    c = _bench().Clocks(0)
    now = time.time()
    c.t0, c.t1 = now, now + 1.0
    c.lines = [_line(now - 0.2, 2062, False), _line(now + 0.1, 1500, True), _line(now + 0.4, 1490, True),
               _line(now + 0.9, 1470, True), _line(now + 1.3, 2062, False)]
    s = c.summary()
    assert s == {"sm_mhz": 1490.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_samples_without_readable_timestamps_all_count():
    c = _bench().Clocks(0)
    now = time.time()
    c.t0, c.t1 = now, now + 1.0
    c.lines = [_line(now - 5, 2062, False).replace("/", "-"), _line(now + 5, 1500, True).replace("/", "-")]
    s = c.summary()
    assert s["samples"] == 2 and s["window"] == "unfiltered" and s["reasons"] == ["sw_power_cap"]


def test_no_samples_gives_no_clock():
    c = _bench().Clocks(0)
    assert c.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
