"""The bench's clock record: nvidia-smi rows sampled during the timed region
are reduced to the median SM clock, the maximum, and every throttle reason
seen active (parsed from a fake sampler process; no GPU needed)."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class FakeProc:
    def __init__(self, text):
        self.text = text

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.text, ""


def sampled(lines):
    s = bench.ClockSampler(0)
    s.proc = FakeProc("\n".join(lines) + "\n")
    return s.stop()


def test_median_clock_and_no_reasons():
    rows = [f"{mhz}, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"
            for mhz in (2070, 2070, 2055, 2070, 1980)]
    c = sampled(rows)
    assert c["sm_mhz"] == 2070 and c["sm_max_mhz"] == 2070 and c["samples"] == 5
    assert c["reasons"] == [] and c["power_w_max"] == 900.5


def test_active_reasons_are_reported():
    rows = ["2070, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
            "1800, 2070, 1390.0, 0x48, Active, Not Active, Not Active, Active",
            "garbage line"]
    c = sampled(rows)
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert c["samples"] == 2 and c["sm_mhz"] == 1935.0


def test_no_sampler_gives_empty_record():
    s = bench.ClockSampler(0)
    s.proc = None
    c = s.stop()
    assert c["sm_mhz"] is None and c["samples"] == 0 and c["reasons"] == []
