"""Pins of the oracle's stochastic tree verification (multi-draft speculative
sampling; Lecture 6 "Optimizing Autoregressive Decode" section 10.3, SpecInfer).

The output law of a node's first token must be the target p, whatever the number
of candidates: checked exactly at V = 16 by driving the oracle over the whole
uniform grid (the accept test is monotone in u, the final draw in floor(u 2^24)),
for candidates drawn i.i.d. from q and for deterministic ("target only")
candidates.  Planted mistakes in the residual update fail the same check."""
import itertools

import numpy as np
import pytest

from oracle import accept as A

GRID = 1 << 24
UMAX = np.float32((GRID - 1) / GRID)


def _first_token(p, q, xs, u):
    """First committed token of a one-level tree: root + children with tokens xs."""
    k = len(xs)
    V = len(p)
    P = np.stack([p] * (k + 1)).astype(np.float32)[None]
    Q = None if q is None else np.stack([q] * (k + 1)).astype(np.float32)[None]
    tok = np.array([[0] + list(xs)])
    parent = np.array([-1] + [0] * k)
    acc, path, com, fin = A.accept_tree_stochastic(P, Q, tok, parent, np.array([u], np.float32))
    return int(com[0, 0]), int(path[0, 0]) if acc[0] > 0 else -1


def _accept_fraction(p, q, xs, j):
    """Fraction of the grid of u[j+1] that accepts child j, earlier children rejected."""
    def accepted(kk):
        u = [0.0] + [UMAX] * j + [kk / GRID] + [0.0] * (len(xs) - j - 1)
        return _first_token(p, q, xs, u)[1] == j + 1      # child j is node j + 1
    lo, hi = 0, GRID
    while lo < hi:
        mid = (lo + hi) // 2
        if accepted(mid):
            lo = mid + 1
        else:
            hi = mid
    return lo / GRID


def _final_law(p, q, xs):
    """Law of the final draw (every child rejected) over the grid of u[0]."""
    out = {}

    def f(kk):
        return _first_token(p, q, xs, [kk / GRID] + [UMAX] * len(xs))[0]

    def runs(lo, hi):
        a, b = f(lo), f(hi)
        if a == b:
            out[a] = out.get(a, 0) + hi - lo + 1
            return
        mid = (lo + hi) // 2
        runs(lo, mid)
        runs(mid + 1, hi)
    runs(0, GRID - 1)
    law = np.zeros(len(p))
    for v, c in out.items():
        law[v] = c / GRID
    return law


def one_level_law(p, q, k):
    """Exact law of the first committed token with k candidates (i.i.d. from q, or all
    ordered k-tuples of distinct tokens weighted uniformly when q is None)."""
    V = len(p)
    law = np.zeros(V)
    if q is None:
        combos = list(itertools.permutations(range(V), k))
        weights = [1.0 / len(combos)] * len(combos)
    else:
        combos = list(itertools.product(range(V), repeat=k))
        weights = [float(np.prod([q[x] for x in xs])) for xs in combos]
    # acceptance of child j depends only on its token and on j (the residual after j
    # rejections depends on q alone), the final law only on k: tabulate once
    acc_tab = {}
    if q is not None:
        # earlier children take the token most likely to be rejected at their step
        # (smallest p_cur / q), so that the rejections the table assumes can happen
        rej, p_cur = [], np.asarray(p, np.float32)
        for j in range(k):
            ratio = np.where(q > 0, p_cur / np.maximum(q, 1e-30), np.inf)
            rej.append(int(np.argmin(ratio)))
            p_cur = A.residual_step(p_cur, q)[0]
        for j in range(k):
            for x in range(V):
                acc_tab[(j, x)] = _accept_fraction(p, q, rej[:j] + [x] + [x] * (k - j - 1), j)
    final_cache = {}
    for xs, w in zip(combos, weights):
        if w == 0:
            continue
        alive = 1.0
        for j, x in enumerate(xs):
            a = acc_tab[(j, x)] if q is not None else _accept_fraction(p, q, list(xs), j)
            law[x] += w * alive * a
            alive *= 1 - a
        if alive > 0:
            key = None if q is not None else tuple(sorted(xs))
            if key not in final_cache:
                final_cache[key] = _final_law(p, q, list(xs))
            law += w * alive * final_cache[key]
    return law


@pytest.mark.parametrize("k", [1, 2, 3])
def test_iid_candidates_law_is_p(k):
    g = np.random.default_rng(k)
    V = 16
    p = g.dirichlet(np.ones(V)).astype(np.float32)
    q = (0.5 * p + 0.5 * g.dirichlet(np.ones(V))).astype(np.float32)
    law = one_level_law(p, q, k)
    np.testing.assert_allclose(law, p, atol=3e-6)


@pytest.mark.parametrize("k", [1, 2, 3])
def test_deterministic_candidates_law_is_p(k):
    g = np.random.default_rng(10 + k)
    V = 8
    p = g.dirichlet(np.ones(V)).astype(np.float32)
    law = one_level_law(p, None, k)
    np.testing.assert_allclose(law, p, atol=3e-6)


def test_first_candidate_acceptance_is_beta_and_more_candidates_accept_more():
    g = np.random.default_rng(4)
    V = 16
    p = g.dirichlet(np.ones(V)).astype(np.float32)
    q = g.dirichlet(np.ones(V)).astype(np.float32)
    beta = np.minimum(p, q).astype(np.float64).sum()
    a1 = sum(q[x] * _accept_fraction(p, q, [x], 0) for x in range(V))
    assert abs(a1 - beta) < 2e-6
    # probability that some candidate is accepted grows with k (1 - P(all rejected))
    def p_any(k):
        tot = 0.0
        for xs in itertools.product(range(V), repeat=k):
            w = float(np.prod([q[x] for x in xs]))
            alive = 1.0
            for j, x in enumerate(xs):
                alive *= 1 - _accept_fraction(p, q, list(xs), j)
            tot += w * (1 - alive)
        return tot
    assert p_any(2) > a1 + 1e-3


@pytest.mark.parametrize("variant", ["no_update", "final_from_p"])
def test_planted_mistakes_break_the_law(monkeypatch, variant):
    g = np.random.default_rng(7)
    V = 16
    p = g.dirichlet(np.ones(V)).astype(np.float32)
    q = (0.5 * p + 0.5 * g.dirichlet(np.ones(V))).astype(np.float32)
    real = A.residual_step
    if variant == "no_update":      # the next sibling is tested against p itself
        monkeypatch.setattr(A, "residual_step", lambda pc, qr: (np.asarray(pc, np.float32).copy(), real(pc, qr)[1]))
    else:                           # the final token drawn from p instead of the residual
        monkeypatch.setattr(A, "residual_step", lambda pc, qr: (real(pc, qr)[0], A.fixed_point_mass(p)))
    law = one_level_law(p, q, 2)
    assert np.abs(law - p).max() > 1e-3


def test_chain_tree_equals_chain_rule():
    """One child per node: the tree rule is Leviathan's chain rule (u index remapped)."""
    g = np.random.default_rng(5)
    for trial in range(40):
        B, gamma, V = 3, int(g.integers(0, 6)), 24
        p = g.dirichlet(np.full(V, 0.5), size=(B, gamma + 1)).astype(np.float32)
        q = g.dirichlet(np.full(V, 0.5), size=(B, gamma)).astype(np.float32)
        q = (0.5 * q + 0.5 * p[:, :gamma]).astype(np.float32)
        x = np.array([[min(int(np.searchsorted(np.cumsum(q[b, i]), g.random())), V - 1) for i in range(gamma)]
                      for b in range(B)]).reshape(B, gamma)
        u = g.random((B, gamma + 1)).astype(np.float32)
        n, com, fin, _ = A.accept_stochastic(p, q, x, u)
        parent = np.arange(-1, gamma)
        tok = np.concatenate([np.zeros((B, 1), np.int64), x], 1)
        qt = np.concatenate([q, np.zeros((B, 1, V), np.float32)], 1)
        ut = np.concatenate([u[:, -1:], u[:, :-1]], 1)
        n2, _, com2, fin2 = A.accept_tree_stochastic(p, qt, tok, parent, ut)
        np.testing.assert_array_equal(n, n2)
        np.testing.assert_array_equal(fin, fin2)
        np.testing.assert_array_equal(com[:, :gamma + 1], com2)


def test_two_level_joint_law_monte_carlo():
    """Two levels, two i.i.d. candidates per node; rows depend only on the token prefix
    (as a model's would).  The empirical law of (first token, second token when the
    first was a candidate) matches the target's p(y1) p(y2 | y1) within 4 sigma."""
    g = np.random.default_rng(11)
    V, n_rounds = 6, 20000
    p0 = g.dirichlet(np.ones(V)).astype(np.float32)
    cond = g.dirichlet(np.ones(V), size=V).astype(np.float32)       # p(y2 | y1)
    q0 = (0.5 * p0 + 0.5 * g.dirichlet(np.ones(V))).astype(np.float32)
    qc = (0.5 * cond + 0.5 * g.dirichlet(np.ones(V), size=V)).astype(np.float32)
    parent = np.array([-1, 0, 0, 1, 1, 2, 2])
    counts = np.zeros((V, V + 1))
    for r in range(n_rounds):
        c1 = [min(int(np.searchsorted(np.cumsum(q0), g.random())), V - 1) for _ in range(2)]
        c2 = [[min(int(np.searchsorted(np.cumsum(qc[t]), g.random())), V - 1) for _ in range(2)] for t in c1]
        tok = np.array([[0, c1[0], c1[1], c2[0][0], c2[0][1], c2[1][0], c2[1][1]]])
        rows = [p0, cond[c1[0]], cond[c1[1]]] + [cond[t] for t in (c2[0][0], c2[0][1], c2[1][0], c2[1][1])]
        qs = [q0, qc[c1[0]], qc[c1[1]]] + [np.zeros(V, np.float32)] * 4
        u = g.random((1, 7)).astype(np.float32)
        acc, path, com, fin = A.accept_tree_stochastic(np.array([rows]), np.array([qs]), tok, parent, u)
        y1 = int(com[0, 0])
        y2 = int(com[0, 1]) if acc[0] >= 1 else V       # V: the round stopped after y1
        counts[y1, y2] += 1
    emp1 = counts.sum(1) / n_rounds
    sd = np.sqrt(p0 * (1 - p0) / n_rounds)
    assert (np.abs(emp1 - p0) < 4 * sd + 1e-9).all()
    # second token given the first, where a second token was produced
    for y1 in range(V):
        m = counts[y1, :V].sum()
        if m < 500:
            continue
        emp = counts[y1, :V] / m
        sd2 = np.sqrt(cond[y1] * (1 - cond[y1]) / m)
        assert (np.abs(emp - cond[y1]) < 4 * sd2 + 1e-9).all(), y1
