"""bench.py prints one JSON line with every key its contract asks for (a
one-layer run of the bench workload, every leg on)."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_has_the_contract_keys():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--layers", "1", "--steps", "3",
           "--warmup", "3", "--cpu-workers", "2"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout[-2000:]
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] >= 3
    assert d["higher_is_better"] is True and d["value"] > 0 and d["gpu_launches"] > 0
    assert d["config"]["workload"]
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] < 2
    e = d["e2e"]
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in e, k
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["timeline"]["stages"] > 0 and e["timeline"]["reading"]
    assert e["pairs"]["n"] >= 1 and e["pairs"]["route_over_probe_median"] > 0
    # the metric's other workloads, each with its resident value, roofline and staged e2e
    wk = d["workloads"]
    assert set(wk) == {"4x31744", "1x262144", "ragged", "1x32768"}
    for name, entry in wk.items():
        assert entry["value"] > 0 and 0 < entry["roofline"]["frac"] < 2, name
        assert entry["e2e"]["value"] > 0 and entry["e2e"]["timeline"]["stages"] > 0, name
    pl = d["e2e_planned"]        # admission-planner window: hot pages resident, the rest staged
    assert pl["value"] > 0 and pl["hot_pages"] > 0 and pl["copied_in_bytes_per_step"] == 0
    bm = d["bus_model"]
    assert len(bm["points"]) == 4 and bm["fit"]["link_GBps"] > 0
    assert "worst_error_pct" in bm and bm["legs"]["per_leg"]
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] == 2 and c["value"] > 0 and c["sample"]
    for k in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert k in d["clocks"], k
