"""The bench's clock record on CPU: nvidia-smi lines (a fake of its CSV
output) are parsed, and the reported clocks come from the samples inside the
timed region, or from the nearest sample on either side when the region is
shorter than the sampling interval."""

import datetime
import time

import bench


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        pass


def _sampler(lines, window):
    c = bench.ClockSampler(0)
    with open(c.f.name, "w") as fh:
        fh.write("\n".join(lines) + "\n")
    c.proc = _Done()
    c.window = list(window)
    return c


def _line(t, sm, cap="Not Active", hw="Not Active"):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{stamp}, 0, {sm}, 2070, 900.0, 0x0, {hw}, Not Active, Not Active, {cap}"


def test_samples_inside_the_timed_region_decide_the_clocks():
    now = time.time()
    lines = [_line(now + 0.05 * k, 2070 if k != 2 else 1500, cap="Active" if k == 5 else "Not Active")
             for k in range(-3, 6)]
    rec = _sampler(lines, (now + 0.01, now + 0.12)).stop()
    assert rec["samples_in_timed_region"] == 2 and rec["samples"] == 2
    assert rec["sm_mhz"] == (2070 + 1500) / 2 and rec["sm_max_mhz"] == 2070
    assert rec["reasons"] == []          # the power-cap sample lies outside the region


def test_short_region_takes_the_neighbouring_samples():
    now = time.time()
    lines = [_line(now + 0.05 * k, 2070, hw="Active" if k == 3 else "Not Active") for k in range(-3, 6)]
    rec = _sampler(lines, (now + 0.101, now + 0.102)).stop()
    assert rec["samples_in_timed_region"] == 0 and rec["samples"] == 2
    assert rec["sm_mhz"] == 2070 and rec["reasons"] == ["hw_slowdown"]   # the sample right after it


def test_lines_without_a_readable_time_still_give_clocks():
    lines = ["garbled-time, 0, 1980, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    rec = _sampler(lines, (None, None)).stop()
    assert rec["sm_mhz"] == 1980 and rec["samples"] == 1
