"""Verify-width planning from a measured step-time curve (host-side scheduling).

"投机解码的性能收支" (speculative-decoding performance accounting), section 四: the
planner ranks each extra candidate by its chance of still being accepted (history
survival probabilities), forms the expected useful progress of a verify budget,
predicts the step time of that budget from a cost table measured on the device,
and picks the budget with the largest progress per unit of step time; rows up to
the execution tier that is paid for anyway verify extra candidates at almost no
cost ("align verify tokens to the graph tier").  Here the tier is the token tile
of the projection kernels: one weight stream serves up to 8, 16, 64 or 128 token
rows (more rows take several 128-row tiles side by side), so the step time is nearly
flat inside a tile.

The trained confidence head that supplies per-candidate survival probabilities
is not part of this library; callers pass survival probabilities (for example
alpha^i from a measured acceptance rate).
"""
from __future__ import annotations

from typing import Dict, Mapping, Sequence, Tuple

TOKEN_TILES = (8, 16, 64, 128)


def survival_iid(alpha: float, n: int) -> list:
    """P(draft i is still accepted) = alpha^i, i = 1..n, for i.i.d. acceptance."""
    return [alpha ** i for i in range(1, n + 1)]


def expected_progress(survival: Sequence[float], width: int) -> float:
    """Expected tokens committed by one chain round of `width` rows: the final token
    (resampled or bonus) always, plus draft i whenever it survives (i < width)."""
    return 1.0 + float(sum(survival[:max(0, width - 1)]))


def token_tile(rows: int) -> int:
    """Token rows one weight stream of the projection kernels covers for `rows` rows."""
    for t in TOKEN_TILES:
        if rows <= t:
            return t
    return TOKEN_TILES[-1] * ((rows + TOKEN_TILES[-1] - 1) // TOKEN_TILES[-1])


def choose_width(step_ms: Mapping[int, float], survival: Sequence[float], batch: int = 1
                 ) -> Tuple[int, Dict[int, float]]:
    """Width W maximising batch * expected_progress(W) / step_ms[W] over the measured
    widths (ties: the smaller width).  Returns (W, {W: tokens per ms})."""
    theta = {w: batch * expected_progress(survival, w) / float(t) for w, t in sorted(step_ms.items())}
    best = max(theta, key=lambda w: (theta[w], -w))
    return best, theta


def align_to_tile(width: int, batch: int, max_width: int) -> int:
    """Largest width <= max_width whose batch * width rows stay in the same token tile
    as batch * width: the extra rows ride on a weight stream that is paid for."""
    tile = token_tile(batch * width)
    w = width
    while w + 1 <= max_width and token_tile(batch * (w + 1)) == tile:
        w += 1
    return w
