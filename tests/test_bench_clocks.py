"""bench.py's clock sampler summarises nvidia-smi rows (index, SM clock, max
SM clock, instantaneous power, throttle flags, power limit) over a time
window: medians, the union of active throttle reasons, and the nearest rows
when the window holds none.  Fed rows here; no GPU, no nvidia-smi."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def row(t, sm, power, cap="Not Active", limit="1400.00"):
    return (t, f"0, {sm}, 2070, {power}, 0x0, Not Active, Not Active, Not Active, {cap}, {limit}")


def sampler_with(rows):
    s = bench.ClockSampler(0)
    s.samples = list(rows)
    return s


def test_window_medians_and_reasons():
    s = sampler_with([row(0.0, 2070, 170.0), row(1.0, 1950, 1380.0, "Active"), row(1.1, 1990, 1366.0),
                      row(1.2, 2010, 1370.0), row(5.0, 2070, 180.0)])
    c = s.summary(1.0, 1.2)
    assert c["window"] == "timed" and c["samples"] == 3
    assert c["sm_mhz"] == 1990 and c["sm_max_mhz"] == 2070
    assert c["power_w"] == 1370.0 and c["power_limit_w"] == 1400.0
    assert c["reasons"] == ["sw_power_cap"]


def test_empty_window_takes_the_nearest_rows():
    s = sampler_with([row(0.0, 2070, 200.0), row(0.1, 2070, 210.0)])
    c = s.summary(10.0, 11.0)
    assert c["window"] == "nearest" and c["samples"] == 2 and c["power_w"] == 205.0 and c["reasons"] == []


def test_unparsable_fields_are_skipped():
    s = sampler_with([row(0.0, 2070, "[N/A]", limit="[N/A]"), row(0.05, 2070, 300.0, limit="[N/A]")])
    c = s.summary(0.0, 0.1)
    assert c["power_w"] == 300.0 and c["power_limit_w"] is None
    assert sampler_with([]).summary(0.0, 1.0)["reasons"] == ["no samples"]
