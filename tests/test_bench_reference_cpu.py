"""The reference arm of bench.py on the CPU: the fp64 oracle timed on the
host cores (the arm the driver runs beside ours) prints one valid JSON line.
A short time budget keeps the test to a few seconds."""

import contextlib
import io
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_line():
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse_args(["--impl", "reference", "--steps", "2", "--warmup", "1",
                             "--cpu-workers", "2"])
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, budget_s=3.0)
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["steps"] == 2 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 2
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
