"""The bench's clock record: nvidia-smi samples are parsed, filtered to the
timed region by their timestamps, and summarised (median SM clock, throttle
reasons seen).  Host logic only: fixed sample lines, no GPU."""
import datetime

import bench

LINES = [
    # timestamp, uuid, clocks.sm, clocks.max.sm, power.draw, reasons bitmask, hw, hw thermal, sw thermal, sw power cap
    "2026/12/02 14:23:35.000, GPU-aaaa, 2070, 2070, 110.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    "2026/12/02 14:23:35.250, GPU-aaaa, 1800, 2070, 1100.0, 0x4, Not Active, Not Active, Not Active, Active",
    "2026/12/02 14:23:35.275, GPU-bbbb, 900, 2070, 300.0, 0x8, Active, Not Active, Not Active, Not Active",
    "2026/12/02 14:23:35.300, GPU-aaaa, 1700, 2070, 1200.0, 0x4, Not Active, Not Active, Not Active, Active",
    "2026/12/02 14:23:35.325, GPU-aaaa, 1750, 2070, 1150.0, 0x4, Not Active, Not Active, Not Active, Active",
    "2026/12/02 14:23:36.000, GPU-aaaa, 2070, 2070, 120.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    "not a sample line",
]


def t(s):
    return datetime.datetime.strptime("2026/12/02 " + s, "%Y/%m/%d %H:%M:%S.%f")


def test_samples_inside_the_timed_region_only():
    r = bench.ClockSampler.parse(LINES, "GPU-aaaa", (t("14:23:35.200"), t("14:23:35.400")))
    assert r["in_timed_region"] == 3 and r["samples"] == 3
    assert r["sm_mhz"] == 1750.0            # median of 1800, 1700, 1750
    assert r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]
    assert r["power_w_max"] == 1200.0


def test_other_gpus_are_ignored():
    # the 900 MHz hw_slowdown sample belongs to another GPU
    r = bench.ClockSampler.parse(LINES, "GPU-aaaa", (t("14:23:35.200"), t("14:23:35.400")))
    assert "hw_slowdown" not in r["reasons"]
    r_all = bench.ClockSampler.parse(LINES, None, (t("14:23:35.200"), t("14:23:35.400")))
    assert "hw_slowdown" in r_all["reasons"] and r_all["samples"] == 4


def test_falls_back_to_every_sample_when_none_is_inside():
    r = bench.ClockSampler.parse(LINES, "GPU-aaaa", (t("14:24:00.000"), t("14:24:01.000")))
    assert r["in_timed_region"] == 0 and r["samples"] == 5
    r = bench.ClockSampler.parse(LINES, "GPU-aaaa", None)
    assert r["in_timed_region"] == 0 and r["samples"] == 5


def test_no_samples():
    r = bench.ClockSampler.parse([], None, None)
    assert r["samples"] == 0 and r["sm_mhz"] is None and r["reasons"] == []
