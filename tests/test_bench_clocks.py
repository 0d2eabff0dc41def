"""Host logic of bench.py's clock record: only samples inside the timed
region decide the reported clock and whether the power cap was seen."""

import tempfile
from datetime import datetime

import bench


def _line(ts, sm, power, cap):
    stamp = datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    act = "Active" if cap else "Not Active"
    return f"{stamp}, 0, {sm}, 2070, {power}, 0x0, Not Active, Not Active, Not Active, {act}\n"


def _sampler(lines, t0, t1):
    s = bench.ClockSampler(0)
    s.proc = object()
    s.out = tempfile.TemporaryFile("w+")
    s.out.write("".join(lines))
    s.t0, s.t1 = t0, t1
    return s


def test_summary_uses_samples_inside_the_timed_region():
    base = 1_800_000_000.0
    lines = [_line(base + 0.00, 1980, 200, False),      # before: idle, boost clock
             _line(base + 0.10, 1450, 1390, True),       # inside: capped
             _line(base + 0.15, 1470, 1385, True),
             _line(base + 0.20, 1500, 1300, False),
             _line(base + 0.40, 2070, 180, False)]       # after
    s = _sampler(lines, base + 0.05, base + 0.30)
    out = s.summary()
    assert out["samples"] == 5 and out["samples_in_timed_region"] == 3
    assert out["power_cap_samples_in_timed_region"] == 2
    assert out["sm_mhz"] == 1470 and out["reasons"] == ["sw_power_cap"]
    assert out["basis"] == "samples inside the timed region"


def test_summary_without_a_sample_inside_says_so():
    base = 1_800_000_000.0
    lines = [_line(base, 2070, 200, False), _line(base + 1.0, 2070, 220, False)]
    out = _sampler(lines, base + 0.2, base + 0.3).summary()
    assert out["samples_in_timed_region"] == 0
    assert out["power_cap_samples_in_timed_region"] == 0
    assert out["basis"].startswith("no sample fell inside")
