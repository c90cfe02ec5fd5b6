"""Pins of the verify-width planner ("投机解码的性能收支", section 四): expected
progress against the closed form of Lecture 6 section 6.3 (the oracle's metric),
the chosen width against brute force, and the token-tile alignment."""
import itertools

import numpy as np
import pytest

from oracle.metrics import expected_tokens_per_round
from speculative_decoding_verify_step_gb300 import planner as P


@pytest.mark.parametrize("alpha", [0.0, 0.3, 0.7, 0.95, 1.0])
def test_expected_progress_is_the_closed_form(alpha):
    for gamma in range(0, 10):
        got = P.expected_progress(P.survival_iid(alpha, 16), gamma + 1)
        assert abs(got - expected_tokens_per_round(alpha, gamma)) < 1e-12


def test_choose_width_bruteforce():
    g = np.random.default_rng(0)
    for _ in range(200):
        widths = sorted(g.choice(np.arange(1, 17), size=g.integers(1, 8), replace=False).tolist())
        step = {w: float(g.uniform(1, 5)) for w in widths}
        surv = np.sort(g.uniform(0, 1, 15))[::-1].tolist()
        B = int(g.integers(1, 65))
        best, theta = P.choose_width(step, surv, B)
        vals = [(B * (1 + sum(surv[:w - 1])) / step[w], -w, w) for w in widths]
        assert best == max(vals)[2]
        assert abs(theta[best] - max(vals)[0]) < 1e-12


def test_flat_and_steep_cost_curves():
    surv = P.survival_iid(0.8, 15)
    flat = {w: 3.0 for w in range(1, 17)}
    assert P.choose_width(flat, surv)[0] == 16          # verify is free: widest
    steep = {w: 3.0 * w for w in range(1, 17)}          # verify costs W decode steps
    assert P.choose_width(steep, surv)[0] == 1          # speculation never pays
    zero = P.survival_iid(0.0, 15)
    assert P.choose_width({1: 3.0, 2: 3.01, 5: 3.1}, zero)[0] == 1


def test_token_tiles_and_alignment():
    assert [P.token_tile(r) for r in (1, 8, 9, 16, 17, 64, 65, 200, 256, 300)] == \
        [8, 8, 16, 16, 64, 64, 128, 256, 256, 384]
    assert P.align_to_tile(5, 1, 16) == 8       # 5 rows -> tile of 8: verify 8
    assert P.align_to_tile(5, 4, 16) == 16      # 20 rows -> tile of 64: 64 rows = width 16
    assert P.align_to_tile(3, 16, 16) == 4      # 48 rows -> tile of 64
    assert P.align_to_tile(9, 1, 12) == 12      # capped by the widest window
    for B, w in itertools.product((1, 2, 3, 7, 16), range(1, 17)):
        a = P.align_to_tile(w, B, 16)
        assert a >= w and P.token_tile(B * a) == P.token_tile(B * w)
