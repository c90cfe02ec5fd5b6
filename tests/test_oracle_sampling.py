"""Pins of the oracle's sampling adjustments (top-k, top-p) and of speculative
sampling on adjusted distributions (Lecture 6 "Optimizing Autoregressive Decode"
section 7.3: adjust p and q the same way and the output follows the adjusted p;
adjusting only p keeps the rule exact at a lower acceptance rate)."""
import itertools

import numpy as np
import pytest

from oracle.accept import accept_stochastic, adjust_probs, adjust_rows
from tests._law import one_position_law

P4 = np.array([0.1, 0.4, 0.2, 0.3], np.float32)   # ranks: token 1, 3, 2, 0


def _close(a, b):
    np.testing.assert_allclose(np.asarray(a, np.float64), b, rtol=0, atol=1e-6)


def test_top_k_hand_values():
    # k = 2 keeps tokens 1 and 3: 0.4 / 0.7 and 0.3 / 0.7
    _close(adjust_probs(P4, 2, 1.0), [0, 4 / 7, 0, 3 / 7])
    _close(adjust_probs(P4, 3, 1.0), [0, 4 / 9, 2 / 9, 3 / 9])
    _close(adjust_probs(P4, 1, 1.0), [0, 1, 0, 0])


def test_top_p_hand_values():
    # cumulative ranked mass 0.4, 0.7, 0.9, 1.0; the crossing token is kept
    _close(adjust_probs(P4, 0, 0.35), [0, 1, 0, 0])
    _close(adjust_probs(P4, 0, 0.5), [0, 4 / 7, 0, 3 / 7])
    _close(adjust_probs(P4, 0, 0.75), [0, 4 / 9, 2 / 9, 3 / 9])
    _close(adjust_probs(P4, 0, 0.95), P4)


def test_top_p_acts_on_the_top_k_renormalised_distribution():
    # k = 2 leaves (4/7, 3/7); 0.55 of that is reached by token 1 alone.  Top-p on
    # the unadjusted p (or top-p first, then top-k) would keep tokens 1 and 3.
    _close(adjust_probs(P4, 2, 0.55), [0, 1, 0, 0])
    _close(adjust_probs(P4, 0, 0.55), [0, 4 / 7, 0, 3 / 7])


def test_equal_probabilities_rank_by_lower_index():
    p = np.full(6, 1 / 6, np.float32)
    _close(adjust_probs(p, 2, 1.0), [0.5, 0.5, 0, 0, 0, 0])
    _close(adjust_probs(p, 0, 0.5), [1 / 3, 1 / 3, 1 / 3, 0, 0, 0])
    p = np.array([0.2, 0.3, 0.2, 0.3], np.float32)
    _close(adjust_probs(p, 3, 1.0), [0.25, 0.375, 0, 0.375])


def test_off_settings_are_the_identity():
    g = np.random.default_rng(0)
    p = g.dirichlet(np.ones(50)).astype(np.float32)
    for k, tp in [(0, 1.0), (50, 1.0), (999, 1.0)]:
        np.testing.assert_array_equal(adjust_probs(p, k, tp), p)


@pytest.mark.parametrize("seed", range(8))
def test_nucleus_is_the_smallest_set_reaching_the_mass_bruteforce(seed):
    """Against enumeration of all 2^10 subsets: the kept set is the smallest set whose
    mass reaches top_p (the most massive one among equally small sets), and top-k
    keeps the k most probable tokens."""
    g = np.random.default_rng(seed)
    V = 10
    p = g.dirichlet(np.full(V, 0.7)).astype(np.float32)
    pd = p.astype(np.float64)
    for tp in (0.3, 0.5, 0.8, 0.9, 0.99):
        best = None
        for n in range(1, V + 1):
            for sub in itertools.combinations(range(V), n):
                m = pd[list(sub)].sum()
                if m >= tp * pd.sum() and (best is None or m > best[1]):
                    best = (set(sub), m)
            if best is not None:
                break
        # a boundary within rounding of the threshold is not a fair test of the set
        if min(abs(best[1] - tp), abs(best[1] - pd[list(best[0])].min() - tp)) < 1e-6:
            continue
        got = adjust_probs(p, 0, tp)
        assert set(np.flatnonzero(got)) == best[0], (tp, got, best)
        np.testing.assert_allclose(got[list(best[0])], pd[list(best[0])] / best[1], rtol=1e-6)
    for k in range(1, V):
        got = adjust_probs(p, k, 1.0)
        assert set(np.flatnonzero(got)) == set(np.argsort(-pd, kind="stable")[:k])


@pytest.mark.parametrize("seed", range(4))
def test_adjusted_rows_are_distributions_proportional_to_p(seed):
    g = np.random.default_rng(seed)
    V = 300
    p = g.dirichlet(np.full(V, 0.3)).astype(np.float32)
    for k, tp in [(1, 1.0), (7, 1.0), (50, 0.9), (0, 0.6), (299, 0.999), (0, 1e-6)]:
        a = adjust_probs(p, k, tp)
        s = np.flatnonzero(a)
        assert abs(a.astype(np.float64).sum() - 1) < 1e-6
        assert len(s) >= 1 and (k == 0 or len(s) <= k)
        ratio = a[s].astype(np.float64) / p[s]
        assert ratio.max() - ratio.min() < 1e-5 * ratio.max()
        # every kept token outranks every dropped one
        assert p[s].min() >= p[np.setdiff1d(np.arange(V), s)].max(initial=0)
    # top-1 and a vanishing nucleus are both the argmax
    am = int(np.argmax(p))
    for k, tp in [(1, 1.0), (0, 1e-9), (3, 1e-9)]:
        a = adjust_probs(p, k, tp)
        assert np.flatnonzero(a).tolist() == [am] and a[am] == 1.0


@pytest.mark.parametrize("k,tp,temp", [(5, 1.0, 1.0), (0, 0.8, 0.5), (6, 0.9, 1.0)])
def test_speculative_sampling_on_adjusted_p_follows_adjusted_p(k, tp, temp):
    """Exact one-position law at V = 16 (every uniform of the 2^24 grid): with p and q
    adjusted alike the output law is the adjusted p and the acceptance is
    sum min(p', q'); with only p adjusted the law is still p' (lower acceptance)."""
    g = np.random.default_rng(k * 10 + int(tp * 10))
    V = 16
    lp = g.normal(size=V) / temp
    p = np.exp(lp - lp.max())
    p = (p / p.sum()).astype(np.float32)
    q = (0.5 * p + 0.5 * g.dirichlet(np.ones(V))).astype(np.float32)
    pa, qa = adjust_probs(p, k, tp), adjust_probs(q, k, tp)
    law, beta, _ = one_position_law(pa, qa)
    np.testing.assert_allclose(law, pa, atol=2e-6)
    assert abs(beta - np.minimum(pa, qa).astype(np.float64).sum()) < 2e-6
    law2, beta2, _ = one_position_law(pa, q)
    np.testing.assert_allclose(law2, pa, atol=2e-6)
    assert abs(beta2 - np.minimum(pa, q).astype(np.float64).sum()) < 2e-6
    assert beta2 <= beta + 1e-9


def test_adjust_rows_per_sequence_settings():
    g = np.random.default_rng(3)
    p = g.dirichlet(np.ones(32), size=(2, 3)).astype(np.float32)
    a = adjust_rows(p, [4, 0], [1.0, 0.7])
    for j in range(3):
        np.testing.assert_array_equal(a[0, j], adjust_probs(p[0, j], 4, 1.0))
        np.testing.assert_array_equal(a[1, j], adjust_probs(p[1, j], 0, 0.7))


def test_top1_sampled_round_is_the_greedy_round():
    """top_k = 1 turns every row into the argmax one-hot: the sampled round then
    accepts exactly the drafts that equal the argmax and commits the argmax."""
    g = np.random.default_rng(9)
    B, gamma, V = 6, 4, 40
    p = g.dirichlet(np.ones(V), size=(B, gamma + 1)).astype(np.float32)
    am = p.argmax(-1)
    x = am[:, :gamma].copy()
    for b in range(B):
        if b < gamma:
            x[b, b] = (x[b, b] + 1) % V
    q = g.dirichlet(np.ones(V), size=(B, gamma)).astype(np.float32)
    u = g.random((B, gamma + 1)).astype(np.float32)
    n, com, tok, _ = accept_stochastic(adjust_rows(p, [1] * B, [1.0] * B), adjust_rows(q, [1] * B, [1.0] * B), x, u)
    for b in range(B):
        nb = b if b < gamma else gamma
        assert n[b] == nb and tok[b] == am[b, nb]
