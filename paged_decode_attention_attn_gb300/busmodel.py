"""Latency model of a decode step on the host-staged route.

"KV-cache engineering", section "Costing the bus before changing anything":
once pinned host memory owns the history, the exact path moves every history
byte over the host link for every generated token, so the step's cost is
written down as a latency model before anything is optimised, and the model is
judged by its worst error against measurement over 32K to 262K tokens.

The model here is the plainest one the staged design supports: with two arena
slots the copy of layer l+1 overlaps the attention of layer l, and at these
sizes the copy is far longer than the attention, so a step costs

    t_step = t_fixed + staged_bytes / link_bandwidth

where staged_bytes is the history the step copies host->device (every layer,
every request) and t_fixed collects the per-step work the copies do not hide
(the last layer's attention and merge, launch and pipeline fill).  ``fit``
estimates the two parameters by least squares from measured (bytes, seconds)
points; ``worst_relative_error`` is the figure the page reports.

Host arithmetic only: the measurements come from the staged decode step.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Iterable, Sequence, Tuple

import numpy as np


@dataclass(frozen=True)
class BusModel:
    fixed_s: float          # per-step time not hidden behind the copies
    link_bytes_per_s: float  # effective host->device bandwidth of the staged copies

    def predict(self, staged_bytes: float) -> float:
        return self.fixed_s + staged_bytes / self.link_bytes_per_s

    def as_dict(self) -> dict:
        return {"fixed_ms": self.fixed_s * 1e3, "link_GBps": self.link_bytes_per_s / 1e9}


def fit(points: Iterable[Tuple[float, float]]) -> BusModel:
    """Least-squares fit of t = a + b * bytes over (bytes, seconds) points."""
    pts = np.asarray(list(points), dtype=np.float64)
    if pts.shape[0] < 2 or np.ptp(pts[:, 0]) == 0:
        raise ValueError("need at least two points with different byte counts")
    A = np.stack([np.ones(len(pts)), pts[:, 0]], axis=1)
    (a, b), *_ = np.linalg.lstsq(A, pts[:, 1], rcond=None)
    if b <= 0:
        raise ValueError("fitted bandwidth is not positive")
    return BusModel(fixed_s=float(a), link_bytes_per_s=float(1.0 / b))


def relative_errors(model: BusModel, points: Sequence[Tuple[float, float]]) -> list:
    return [abs(model.predict(x) - t) / t for x, t in points]


def worst_relative_error(model: BusModel, points: Sequence[Tuple[float, float]]) -> float:
    return max(relative_errors(model, points))


def staged_bytes_per_step(lengths, n_layers: int, row_bytes: int) -> int:
    """History bytes a whole-history staged step copies: every layer's rows of
    every request except the new token's row (produced on the device and only
    written back)."""
    return sum(max(0, int(L) - 1) for L in lengths) * row_bytes * n_layers
