"""The staged-route latency model: fitting and error arithmetic (no GPU)."""

import numpy as np
import pytest

from paged_decode_attention_attn_gb300 import busmodel as bm


def test_fit_recovers_exact_parameters():
    truth = bm.BusModel(fixed_s=0.8e-3, link_bytes_per_s=211e9)
    xs = [2.1e9, 4.3e9, 8.6e9, 17.2e9]
    pts = [(x, truth.predict(x)) for x in xs]
    m = bm.fit(pts)
    assert m.fixed_s == pytest.approx(truth.fixed_s, rel=1e-9)
    assert m.link_bytes_per_s == pytest.approx(truth.link_bytes_per_s, rel=1e-9)
    assert bm.worst_relative_error(m, pts) < 1e-9


def test_worst_error_is_the_largest_relative_miss():
    m = bm.BusModel(fixed_s=0.0, link_bytes_per_s=1e9)
    pts = [(1e9, 1.0), (2e9, 2.2), (4e9, 3.8)]
    errs = bm.relative_errors(m, pts)
    assert errs == pytest.approx([0.0, 0.2 / 2.2, 0.2 / 3.8])
    assert bm.worst_relative_error(m, pts) == pytest.approx(0.2 / 2.2)


def test_fit_is_least_squares_on_noisy_points():
    rng = np.random.default_rng(0)
    xs = np.linspace(1e9, 2e10, 9)
    ts = 1e-3 + xs / 2e11 + rng.normal(0, 1e-4, xs.size)
    m = bm.fit(zip(xs, ts))
    A = np.stack([np.ones_like(xs), xs], 1)
    a, b = np.linalg.lstsq(A, ts, rcond=None)[0]
    assert m.fixed_s == pytest.approx(a) and m.link_bytes_per_s == pytest.approx(1 / b)


def test_degenerate_inputs_are_refused():
    with pytest.raises(ValueError):
        bm.fit([(1e9, 1.0)])
    with pytest.raises(ValueError):
        bm.fit([(1e9, 1.0), (1e9, 2.0)])
    with pytest.raises(ValueError):
        bm.fit([(1e9, 2.0), (2e9, 1.0)])      # time falling with bytes


def test_staged_bytes_counts_history_without_the_new_row():
    assert bm.staged_bytes_per_step([31744] * 4, 16, 4096) == 4 * 31743 * 4096 * 16


def test_bench_predictions_use_single_steps_on_a_free_link():
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    model = bm.BusModel(fixed_s=0.001, link_bytes_per_s=200e9)
    legs = {"a": {"staged_bytes_per_step": 2_000_000_000,          # predicts 11 ms
                  "pairs": {"step_ms": [11.0, 40.0, 11.5, 30.0], "step_ms_median": 20.75,
                            "stage_min_GBps": [210.0, 60.0, 205.0, 80.0]}},
            "b": {"staged_bytes_per_step": 1_000_000_000,
                  "pairs": {"step_ms": [50.0], "step_ms_median": 50.0,
                            "stage_min_GBps": [50.0]}}}
    out = bench.bus_predictions(model, legs, best_stage=211.0)
    a = out["per_leg"]["a"]
    assert a["pairs_used"] == 2 and a["measured_ms"] == 11.25          # the two free-link pairs
    assert a["predicted_ms"] == 11.0
    assert a["error_pct"] == round(100 * (11.0 - 11.25) / 11.25, 3)
    assert out["per_leg"]["b"]["pairs_used"] == 0                       # no free-link pair
    assert out["worst_abs_error_pct"] == abs(a["error_pct"])
