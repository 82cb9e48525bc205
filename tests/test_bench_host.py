"""Host logic of bench.py that needs no GPU: the clock-sample window, the traffic
provenance digests and the --slab-cap option."""
import datetime
import importlib.util
import os
import time

import pytest

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


def test_traffic_figures_go_null_when_the_kernel_source_changes(monkeypatch):
    b = _bench()
    wl = b.wk.LINEAR_HEADLINE
    for kind, (names, _) in b.TRAFFIC_SOURCES.items():
        now = b.source_digest(names)
        assert len(now) == 16 and int(now, 16) >= 0
        # pretend the counters were taken on exactly the current sources
        monkeypatch.setitem(b.TRAFFIC_SOURCES, kind, (names, now))
    assert b.FWD_GEMM_TRAFFIC_BYTES(wl) is not None
    assert b.LOGITS_TRAFFIC_BYTES(b.wk.LOGITS_MEMBOUND, "backward") is not None
    # any other digest means the kernel changed after the capture: no traffic figure
    names, _ = b.TRAFFIC_SOURCES["gemm"]
    monkeypatch.setitem(b.TRAFFIC_SOURCES, "gemm", (names, "0" * 16))
    assert b.FWD_GEMM_TRAFFIC_BYTES(wl) is None
    names, _ = b.TRAFFIC_SOURCES["rows"]
    monkeypatch.setitem(b.TRAFFIC_SOURCES, "rows", (names, "0" * 16))
    assert b.LOGITS_TRAFFIC_BYTES(b.wk.LOGITS_MEMBOUND, "fused") is None


def test_slab_cap_option():
    # --slab-cap: the library default (0), one slab (SIZE_MAX) or a byte count
    bench = _bench()
    assert bench.parse_slab_cap("default") == 0
    assert bench.parse_slab_cap("uncapped") == (1 << 64) - 1
    assert bench.parse_slab_cap("67108864") == 64 << 20
    for bad in ("0", "-5", "lots"):
        with pytest.raises(ValueError):
            bench.parse_slab_cap(bad)
    assert bench.slab_cap_label(0).startswith("library default")
    assert bench.slab_cap_label(bench.SLAB_UNCAPPED) == "uncapped"
    assert bench.slab_cap_label(64 << 20) == 64 << 20
