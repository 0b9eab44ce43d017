"""The staged legs' timeline arithmetic (bench.timeline_stats) on fake
events with known times: copy time counts from when the H2D stream reached
the stage and the slot's previous readers were done; idle time before a
stage is split into host gap and slot wait.  No GPU needed."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class Ev:
    def __init__(self, t):
        self.t = t

    def elapsed_time(self, other):
        return other.t - self.t


def stage(s0, s1, c2, c3, d4):
    return [Ev(s0), Ev(s1), Ev(c2), Ev(c3), Ev(d4)]


def test_timeline_splits_h2d_time_into_copy_slot_wait_and_host_gap():
    # 2 slots, 1,000,000 bytes per stage, 4 stages (2 steps of 2 stages).
    ev = [
        stage(0.0, 1.0, 1.0, 1.5, 1.6),     # copy 1.0
        stage(1.0, 2.0, 2.0, 2.5, 2.6),     # copy 1.0, no gap
        stage(2.5, 3.0, 3.0, 3.2, 3.3),     # host gap 0.5; slot readers done at 1.6: copy 0.5
        stage(3.0, 5.0, 5.0, 5.5, 5.6),     # slot readers (stage 1) done at 2.6 < 3.0: copy 2.0
    ]
    r = bench.timeline_stats(ev, 2, [1_000_000, 1_000_000], steps=2)
    assert r["stages"] == 4
    assert r["copy_ms"] == {"median": 1.0, "min": 0.5, "max": 2.0}
    assert r["host_gap_ms_per_step"] == pytest.approx(0.25)
    assert r["slot_wait_ms_per_step"] == 0.0
    assert r["copy_GBps"]["max"] == pytest.approx(2.0)     # 1 MB in 0.5 ms
    assert r["copy_GBps"]["min"] == pytest.approx(0.5)     # 1 MB in 2 ms
    assert r["h2d_region_ms"] == 5.0
    assert r["h2d_time_split"]["copying"] == pytest.approx(4.5 / 5)
    assert r["h2d_time_split"]["host_gap"] == pytest.approx(0.5 / 5)
    assert r["attention_ms_median"] == pytest.approx(0.5)


def test_timeline_counts_a_slot_wait_when_the_previous_reader_is_late():
    ev = [
        stage(0.0, 1.0, 1.0, 4.0, 4.1),     # attention of stage 0 runs late (ends 4.0, wb 4.1)
        stage(1.0, 2.0, 4.0, 4.5, 4.6),     # compute waits 0 (busy with stage 0 until 4.0)
        stage(2.0, 5.1, 5.1, 5.5, 5.6),     # waits for stage 0's readers until 4.1: copy 1.0
    ]
    r = bench.timeline_stats(ev, 2, [2_000_000], steps=1)
    assert r["slot_wait_ms_per_step"] == pytest.approx(2.1)
    assert r["copy_ms"]["max"] == pytest.approx(1.0)
    assert r["compute_wait_ms_per_step"] == pytest.approx(0.6)   # 4.5 -> 5.1


def test_timeline_reading_names_the_bound():
    r = bench.timeline_reading({"h2d_time_split": {"copying": 0.999, "slot_wait": 0.0005,
                                                    "host_gap": 0.0005},
                                "copy_GBps": {"median": 210.0, "min": 31.0}})
    assert r.startswith("link-bound") and "31.0 GB/s" in r
    r = bench.timeline_reading({"h2d_time_split": {"copying": 0.7, "slot_wait": 0.05,
                                                    "host_gap": 0.25},
                                "copy_GBps": {"median": 210.0, "min": 200.0}})
    assert "waiting for the host" in r and "25.0%" in r


def test_timeline_accounts_for_stages_that_copied_slowly():
    # 1 slot, 10 MB per stage: three stages at 10 GB/s (1 ms) and one at
    # 2.5 GB/s (4 ms): one slow stage, 3 ms beyond the fastest stage's rate.
    ev = [
        stage(0.0, 1.0, 1.0, 1.1, 1.2),
        stage(1.2, 2.2, 2.2, 2.3, 2.4),
        stage(2.4, 6.4, 6.4, 6.5, 6.6),
        stage(6.6, 7.6, 7.6, 7.7, 7.8),
    ]
    r = bench.timeline_stats(ev, 1, [10_000_000], steps=2)
    slow = r["slow_stages"]
    assert slow["n"] == 1 and slow["of"] == 4
    assert slow["fastest_stage_GBps"] == pytest.approx(10.0)
    assert slow["below_GBps"] == pytest.approx(9.0)
    assert slow["rates_GBps"] == [2.5]
    assert slow["excess_ms_per_step"] == pytest.approx(1.5)     # 3 ms over 2 steps
    r["h2d_time_split"] = {"copying": 0.99, "slot_wait": 0.0, "host_gap": 0.01}
    text = bench.timeline_reading(r)
    assert "1 of 4 stages" in text and "1.5 ms" in text


def test_free_link_rate_uses_single_steps_whose_stages_all_ran_at_link_rate():
    # (step seconds, probe GB/s, slowest stage GB/s); the leg's fastest stage 210
    pairs = [(0.040, 211.0, 205.0), (0.080, 211.0, 40.0), (0.042, 211.0, 200.0)]
    tl = {"copy_GBps": {"max": 210.0}}
    assert bench.free_link_rate(8.4e9, pairs, tl) == round(8.4e9 / 0.041 / 1e9, 2)
    assert bench.free_link_rate(8.4e9, [(0.08, 211.0, 40.0)], tl) is None
