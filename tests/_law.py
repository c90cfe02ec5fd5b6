"""Exact one-round output law of the oracle's acceptance rule, by enumeration.

Drives `oracle.accept.accept_stochastic` itself over every value of the
uniform grid the rule can see (u = k / 2^24 for the accept test and for the
final draw), using monotonicity to count whole runs of the grid at once:
the accept test fl32(u*q) < p is monotone in u, and the integer inverse-CDF
draw is monotone in floor(u * 2^24).  Nothing of the rule is re-typed here.
"""
from __future__ import annotations

import numpy as np

from oracle.accept import accept_stochastic

GRID = 1 << 24


def _u(k: int) -> np.float32:
    return np.float32(k / GRID)


def _round(p, q, x, k0, k1, **kw):
    V = len(p)
    P = np.stack([p, p]).astype(np.float32)[None]            # rows 0 and 1
    Q = np.asarray(q, np.float32).reshape(1, 1, V)
    n, committed, _, _ = accept_stochastic(P, Q, np.array([[x]]),
                                           np.array([[_u(k0), _u(k1)]], np.float32), **kw)
    return int(n[0]), int(committed[0, 0])


def _count_runs(f, lo, hi, out):
    """f monotone non-decreasing on [lo, hi]; add the number of k giving each value."""
    a, b = f(lo), f(hi)
    if a == b:
        out[a] = out.get(a, 0) + (hi - lo + 1)
        return
    mid = (lo + hi) // 2
    _count_runs(f, lo, mid, out)
    _count_runs(f, mid + 1, hi, out)


def one_position_law(p, q, **kw):
    """Returns (law [V] of the first committed token, P(accept), residual law given x).

    p, q: float32 [V].  kw are passed to accept_stochastic (planted variants).
    """
    p = np.asarray(p, np.float32)
    q = np.asarray(q, np.float32)
    V = len(p)
    law = np.zeros(V)
    p_acc = 0.0
    res_laws = {}
    for x in range(V):
        if q[x] == 0:
            continue
        # number of grid points k with the draft accepted (a prefix of the grid)
        lo, hi = 0, GRID                     # acceptance holds for k < k_star
        while lo < hi:
            mid = (lo + hi) // 2
            if _round(p, q, x, mid, 0, **kw)[0] == 1:
                lo = mid + 1
            else:
                hi = mid
        k_star = lo
        a = k_star / GRID
        law[x] += q[x] * a
        p_acc += q[x] * a
        if k_star < GRID:
            counts = {}
            _count_runs(lambda m: _round(p, q, x, GRID - 1, m, **kw)[1], 0, GRID - 1, counts)
            rl = np.zeros(V)
            for v, c in counts.items():
                rl[v] = c / GRID
            res_laws[x] = rl
            law += q[x] * (1 - a) * rl
    return law, p_acc, res_laws
