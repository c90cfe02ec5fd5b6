"""Pins of the oracle's acceptance rules against what the pages and mathematics fix."""
import numpy as np
import pytest

from oracle import accept as A
from oracle import metrics as M
from tests._law import one_position_law


def tv(a, b):
    return 0.5 * float(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)).sum())


# --------------------------------------------------------------- worked examples
def test_exercise3_exact_law(golden):
    g = golden("ex3_one_position_law.json")
    p, q = np.array(g["p"], np.float32), np.array(g["q"], np.float32)
    law, beta, res = one_position_law(p, q)
    assert beta == pytest.approx(g["beta"], abs=1e-6)
    assert 1 - tv(p, q) == pytest.approx(g["beta"], abs=1e-6)
    assert tv(p, q) == pytest.approx(g["tv"], abs=1e-6)
    for x, rl in res.items():              # the residual is (1, 0, 0) whatever x was
        np.testing.assert_allclose(rl, g["residual_normalised"], atol=1e-9)
    np.testing.assert_allclose(law, g["output_law"], atol=1e-6)


def test_exercise4_resample_from_p_is_detected(golden):
    g = golden("ex4_resample_from_p_variant.json")
    p, q = np.array(g["p"], np.float32), np.array(g["q"], np.float32)
    # planted mistake: redraw from p after a rejection instead of the residual
    law, _, _ = one_position_law(p, q, residual_fn=lambda pr, qr: pr)
    np.testing.assert_allclose(law, g["output_law"], atol=1e-6)
    assert tv(law, p) == pytest.approx(g["tv_to_p"], abs=1e-6)
    good, _, _ = one_position_law(p, q)
    assert tv(good, p) < 1e-6


def test_deterministic_reject_variant_is_detected():
    # planted mistake: reject whenever q(x) > p(x), with no randomness
    p = np.array([0.5, 0.3, 0.2], np.float32)
    q = np.array([0.2, 0.6, 0.2], np.float32)
    law, beta, _ = one_position_law(p, q, accept_fn=lambda u, qx, px: qx <= px)
    # accepts a and c (0.4 of the mass), residual is (1,0,0): law (0.8, 0, 0.2)
    np.testing.assert_allclose(law, [0.8, 0.0, 0.2], atol=1e-6)
    assert tv(law, p) > 0.25


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_exact_law_equals_p_v16(seed):
    """Sections 7.1/7.2: the one-round output law is p; P(accept) = sum min(p,q) = 1 - TV."""
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.ones(16)).astype(np.float32)
    q = rng.dirichlet(np.ones(16) * 0.5).astype(np.float32)
    law, beta, _ = one_position_law(p, q)
    assert beta == pytest.approx(float(np.minimum(p, q).sum()), abs=2e-6)
    assert beta == pytest.approx(1 - tv(p, q), abs=2e-6)
    np.testing.assert_allclose(law, p, atol=2e-6)
    bad, _, _ = one_position_law(p, q, residual_fn=lambda pr, qr: pr)
    assert tv(bad, p) > 1e-3


# ------------------------------------------------------------- multi-position MC
def _markov(seed, V=16):
    rng = np.random.default_rng(seed)
    P = rng.dirichlet(np.ones(V) * 0.7, size=V)
    Q = rng.dirichlet(np.ones(V) * 0.7, size=V)
    return P.astype(np.float32), Q.astype(np.float32)


def _draw(rows, r):
    c = np.cumsum(rows.astype(np.float64), axis=1)
    c[:, -1] = 1.0
    return (c < r[:, None]).sum(axis=1)


def _two_tokens(P, Q, N, gamma, seed, **kw):
    """First two committed tokens of N independent chains, starting from token 0."""
    rng = np.random.default_rng(seed)
    V = P.shape[0]
    out = np.full((N, 2), -1, np.int64)
    pending = np.zeros(N, np.int64)
    have = np.zeros(N, np.int64)
    accepted_total, proposed_total = 0, 0
    for _ in range(3):
        need = np.nonzero(have < 2)[0]
        if len(need) == 0:
            break
        B = len(need)
        toks = np.zeros((B, gamma + 1), np.int64)
        toks[:, 0] = pending[need]
        for i in range(1, gamma + 1):
            toks[:, i] = _draw(Q[toks[:, i - 1]], rng.random(B))
        p = P[toks]                                   # row j: p after token j
        q = Q[toks[:, :gamma]]
        u = rng.random((B, gamma + 1)).astype(np.float32)
        n, committed, _, _ = A.accept_stochastic(p, q, toks[:, 1:], u, **kw)
        accepted_total += int(n.sum())
        proposed_total += B * gamma
        for r, b in enumerate(need):
            for t in committed[r, :n[r] + 1]:
                if have[b] < 2:
                    out[b, have[b]] = t
                    have[b] += 1
            pending[b] = committed[r, n[r]]
    return out, accepted_total, proposed_total


def test_markov_joint_law_of_two_tokens():
    """Section 7.5's experiment at V=16, gamma=3: the joint law of the first two
    output tokens equals the target's; both wrong variants are far off."""
    P, Q = _markov(7)
    V, N, gamma = 16, 400_000, 3
    exact = np.outer(P[0], np.ones(V)) * P          # P(a) P(b | a)
    out, _, _ = _two_tokens(P, Q, N, gamma, seed=11)
    emp = np.bincount(out[:, 0] * V + out[:, 1], minlength=V * V).reshape(V, V) / N
    # sampling noise: E[TV] ~ 0.5 * sum sqrt(2 p / (pi N)) (about 0.008 here)
    noise = 0.5 * np.sqrt(2 * exact / (np.pi * N)).sum()
    assert tv(emp, exact) < 2.0 * noise
    bad, _, _ = _two_tokens(P, Q, N, gamma, seed=11, residual_fn=lambda pr, qr: pr)
    emp_bad = np.bincount(bad[:, 0] * V + bad[:, 1], minlength=V * V).reshape(V, V) / N
    assert tv(emp_bad, exact) > 4.0 * noise
    det, _, _ = _two_tokens(P, Q, N, gamma, seed=11, accept_fn=lambda u, qx, px: qx <= px)
    emp_det = np.bincount(det[:, 0] * V + det[:, 1], minlength=V * V).reshape(V, V) / N
    assert tv(emp_det, exact) > 4.0 * noise


def test_measured_acceptance_equals_beta():
    """Per-draft acceptance of the first draft equals E_x0[sum min(p, q)]."""
    P, Q = _markov(3)
    rng = np.random.default_rng(5)
    N = 400_000
    toks = np.zeros((N, 2), np.int64)
    toks[:, 1] = _draw(Q[toks[:, 0]], rng.random(N))
    u = rng.random((N, 2)).astype(np.float32)
    n, _, _, _ = A.accept_stochastic(P[toks], Q[toks[:, :1]], toks[:, 1:], u)
    beta = float(np.minimum(P[0], Q[0]).sum())
    assert n.mean() == pytest.approx(beta, abs=4 * np.sqrt(beta * (1 - beta) / N))


# ---------------------------------------------------------- tokens per round
def _iid_rounds(alpha, gamma, N, seed):
    """V=2 construction with per-draft acceptance exactly alpha: q = (1, 0), p = (alpha, 1-alpha)."""
    p_row = np.array([alpha, 1 - alpha], np.float32)
    q_row = np.array([1.0, 0.0], np.float32)
    p = np.broadcast_to(p_row, (N, gamma + 1, 2)).copy()
    q = np.broadcast_to(q_row, (N, gamma, 2)).copy()
    x = np.zeros((N, gamma), np.int64)
    u = np.random.default_rng(seed).random((N, gamma + 1)).astype(np.float32)
    n, committed, _, _ = A.accept_stochastic(p, q, x, u)
    return n + 1


@pytest.mark.parametrize("ex,alpha,gamma,expect", [("ex5", 0.75, 7, 3.60), ("ex7", 0.7, 3, 2.533)])
def test_tokens_per_round(golden, ex, alpha, gamma, expect):
    g = golden("tokens_per_round_exercises.json")[ex]
    assert (g["alpha"], g["gamma"], g["tokens_per_round"]) == (alpha, gamma, expect)
    closed = M.expected_tokens_per_round(alpha, gamma)
    digits = len(str(expect).split(".")[1])
    assert abs(closed - expect) <= 0.5 * 10 ** -digits
    tpr = _iid_rounds(alpha, gamma, 400_000, seed=gamma)
    assert tpr.mean() == pytest.approx(closed, abs=4 * tpr.std() / np.sqrt(len(tpr)))


def test_tokens_per_round_exercise_numbers(golden):
    g = golden("tokens_per_round_exercises.json")
    e5 = g["ex5"]
    c = (M.expected_tokens_per_round(e5["alpha"], e5["gamma"]) / e5["measured_speedup"] - 1) / e5["gamma"]
    assert abs(c - e5["implied_c"]) <= 0.0005
    e6 = g["ex6"]
    for gm, s in zip(e6["gamma"], e6["speedup"]):
        assert abs(M.walltime_speedup(e6["alpha"], gm, e6["c"]) - s) <= 0.005
    e7 = g["ex7"]
    assert abs(M.compute_factor(e7["alpha"], e7["gamma"], 0.0) - e7["factor_chat0"]) <= 0.005
    assert abs(M.compute_factor(e7["alpha"], e7["gamma"], 0.1) - e7["factor_chat01"]) <= 0.005
    e11 = g["ex11"]
    assert abs(1 / e11["tokens_per_forward"] - e11["weight_read_ratio"]) <= 0.005


def test_accounting_metrics_example(golden):
    g = golden("accounting_metrics_example.json")
    c = M.Counters()
    c.record_round(gamma=g["proposed_drafts"], accepted=[g["accepted_drafts"]])
    assert c.verify_steps == g["verify_steps"]
    assert c.committed == g["accepted_drafts"] + g["bonus_tokens"]
    assert c.strict_accept_rate == pytest.approx(g["strict_accept_rate"])
    assert c.accept_length == pytest.approx(g["accept_length"])


def test_verify_cost_division(golden):
    g = golden("verify_cost_division.json")
    s = M.speedup_gamma1(g["p"], g["t_decode_ms"], g["t_verify_ms"], g["t_draft_ms"])
    assert abs(s * 1000 / g["t_decode_ms"] - g["tok_per_s"]) < 0.5
    assert abs((1 + g["p"]) / (g["t_verify_ms"] + g["t_draft_ms"]) - g["tokens_per_ms"]) < 0.0005
    be = M.breakeven_verify(g["p"], g["t_decode_ms"], g["t_draft_ms"])
    assert abs(be - g["breakeven_verify_ms"]) < 0.05
    assert abs(be / g["t_decode_ms"] - g["breakeven_ratio"]) < 0.005
    s3 = g["section3"]
    for k in ("wrong", "right"):
        tps = 1000 * (1 + s3["p"]) / (2 * s3[f"{k}_t_decode_ms"] + s3["t_draft_ms"])
        assert abs(tps - s3[f"{k}_tok_s"]) < 0.05
        # the page rounds either the tok/s figure or the ratio first; one of them
        # must reproduce its printed ratio to half a unit of the last digit
        r_exact = tps / s3["baseline_tok_s"]
        r_rounded = s3[f"{k}_tok_s"] / s3["baseline_tok_s"]
        assert min(abs(r_exact - s3[f"{k}_ratio"]), abs(r_rounded - s3[f"{k}_ratio"])) < 0.0005
    # two full passes can never win at one guess per round: (1+p)/2 <= 1
    for p in (0.0, 0.5, 1.0):
        assert M.speedup_gamma1(p, 1.0, 2.0, 0.0) <= 1.0


# ------------------------------------------------------------------- greedy
def test_greedy_cumprod_semantics():
    V = 8
    logits = np.zeros((1, 4, V))
    am = [3, 5, 1, 7]
    for j, a in enumerate(am):
        logits[0, j, a] = 1.0
    for x, n in [([3, 5, 1], 3), ([3, 4, 1], 1), ([2, 5, 1], 0), ([3, 5, 0], 2)]:
        acc, com, bonus = A.accept_greedy(logits, np.array([x]))
        assert acc[0] == n
        assert list(com[0, :n]) == x[:n]
        assert com[0, n] == am[n] == bonus[0]
        assert (com[0, n + 1:] == -1).all()


def test_greedy_tie_lowest_index():
    logits = np.zeros((1, 1, 6))
    logits[0, 0, [2, 4]] = 3.0
    _, com, bonus = A.accept_greedy(logits, np.zeros((1, 0), np.int64))
    assert bonus[0] == 2


def test_greedy_is_the_temperature_zero_limit():
    """Section 7.4: at T -> 0 the stochastic rule commits exactly the greedy tokens."""
    rng = np.random.default_rng(4)
    B, g, V = 64, 3, 12
    logits = rng.normal(size=(B, g + 1, V)) * 3
    am = logits.argmax(-1)
    x = np.where(rng.random((B, g)) < 0.6, am[:, :g], rng.integers(0, V, (B, g)))
    p = A.target_probs(logits, 1e-4)            # one-hot in float32
    q = np.zeros((B, g, V), np.float32)
    q[np.arange(B)[:, None], np.arange(g)[None], x] = 1.0
    u = rng.random((B, g + 1)).astype(np.float32)
    n_s, com_s, _, _ = A.accept_stochastic(p, q, x, u)
    n_g, com_g, _ = A.accept_greedy(logits, x)
    np.testing.assert_array_equal(n_s, n_g)
    np.testing.assert_array_equal(com_s, com_g)


# ------------------------------------------------------------- integer draw
def test_draw_index_bruteforce():
    rng = np.random.default_rng(9)
    for _ in range(200):
        V = int(rng.integers(1, 40))
        r = (rng.random(V) * (rng.random(V) < 0.7)).astype(np.float32)
        R = A.fixed_point_mass(r)
        u = np.float32(rng.random())
        S = sum(int(v) for v in R)
        got = A.draw_index(R, u)
        if S == 0:
            assert got == -1
            continue
        m = int(np.floor(float(u) * 2 ** 24))
        t = m * S // 2 ** 24
        run = 0
        for v in range(V):
            run += int(R[v])
            if run > t:
                break
        assert got == v and R[v] > 0
        assert A.draw_index_rows(R[None], np.array([u]))[0] == got


def test_draw_index_rows_no_overflow():
    # masses near the 2^58 bound: the split product must stay exact
    V = 1 << 17
    r = np.ones(V, np.float32)
    R = A.fixed_point_mass(r)
    for u in [0.0, 0.5, 1 - 2 ** -24, 0.123456789]:
        assert A.draw_index_rows(R[None], np.array([u], np.float32))[0] == A.draw_index(R, u)


def test_fixed_point_mass_exact():
    r = np.array([1.0, 0.5, 2 ** -40, 2 ** -41, 0.0, 0.3], np.float32)
    R = A.fixed_point_mass(r)
    assert list(R[:5]) == [2 ** 40, 2 ** 39, 1, 0, 0]
    assert int(R[5]) == int(np.floor(float(np.float32(0.3)) * 2 ** 40))


def test_zero_residual_falls_back_to_p():
    # p == q: every draft accepted except when fl32(u q) rounds up to q; force a
    # rejection through the planted accept_fn and check the fallback draw from p
    p = np.array([[[0.25, 0.75], [0.5, 0.5]]], np.float32)
    q = np.array([[[0.25, 0.75]]], np.float32)
    n, com, tok, zero = A.accept_stochastic(p, q, np.array([[1]]), np.array([[0.9, 0.1]], np.float32),
                                            accept_fn=lambda u, qx, px: np.zeros_like(u, bool))
    assert n[0] == 0 and zero[0] and tok[0] == 0      # floor(0.1*2^24)*S>>24 lands in token 0


def test_massless_target_row_gives_token_0():
    """A target row with no mass on the 2^-40 grid (all zeros, or every entry below
    2^-40) is not a distribution; the draw returns token 0 by the stated reading,
    in the chain (after a rejection, and as the bonus) and in the tree."""
    V = 6
    for row in (np.zeros(V, np.float32), np.full(V, 2.0 ** -42, np.float32)):
        p = np.stack([row, row])[None]                                  # [1, 2, V]
        q = np.full((1, 1, V), 1.0 / V, np.float32)
        for u_last in (0.0, 0.37, 0.999):
            u = np.array([[0.5, u_last]], np.float32)
            n, com, tok, zero = A.accept_stochastic(p, q, np.array([[3]]), u)   # p(x) = 0: rejected
            assert n[0] == 0 and zero[0] and tok[0] == 0 and com[0].tolist() == [0, -1]
            n, com, tok, _ = A.accept_stochastic(p, q, np.array([[3]]), u,
                                                 accept_fn=lambda u_, qx, px: np.ones_like(u_, bool))
            assert n[0] == 1 and tok[0] == 0 and com[0].tolist() == [3, 0]
            pt = np.stack([row, row])[None]
            for qq in (None, np.full((1, 2, V), 1.0 / V, np.float32)):
                acc, path, com, fin = A.accept_tree_stochastic(pt, qq, np.array([[1, 4]]), np.array([-1, 0]),
                                                               np.array([[u_last, 0.5]], np.float32))
                assert acc[0] == 0 and fin[0] == 0 and com[0, 0] == 0
    # one token with grid mass is drawn whatever u is
    row = np.zeros(V, np.float32)
    row[4] = 2.0 ** -40
    p = np.stack([row, row])[None]
    for u_last in (0.0, 0.5, 0.999):
        _, _, tok, _ = A.accept_stochastic(p, np.full((1, 1, V), 1.0 / V, np.float32), np.array([[3]]),
                                           np.array([[0.5, u_last]], np.float32))
        assert tok[0] == 4


# -------------------------------------------------------------------- tree
def _brute_tree(logits, tok, parent):
    N = len(parent)
    best, best_depth = 0, 0
    depth = A.tree_depths(parent)
    for c in range(1, N):
        ok, v = True, c
        while parent[v] >= 0:
            pa = parent[v]
            if tok[v] != np.argmax(logits[pa]):
                ok = False
                break
            v = pa
        if ok and depth[c] > best_depth:
            best, best_depth = c, depth[c]
    return best, best_depth


def test_tree_walk_bruteforce():
    rng = np.random.default_rng(2)
    for trial in range(300):
        N = int(rng.integers(1, 16))
        parent = np.array([-1] + [int(rng.integers(0, c)) for c in range(1, N)])
        V = 6
        logits = rng.normal(size=(1, N, V))
        tok = rng.integers(0, V, (1, N))
        # no two siblings share a token: the matched path is then unique
        for v in range(N):
            kids = [c for c in range(1, N) if parent[c] == v]
            perm = rng.permutation(V)
            for i, c in enumerate(kids[:V]):
                tok[0, c] = perm[i]
            if len(kids) > V:
                continue
        if any(len([c for c in range(1, N) if parent[c] == v]) > V for v in range(N)):
            continue
        acc, path, com, bonus = A.accept_tree_greedy(logits, tok, parent)
        node, d = _brute_tree(logits[0], tok[0], parent)
        assert acc[0] == d
        if d:
            assert path[0, d - 1] == node
        assert bonus[0] == np.argmax(logits[0, node])
        assert com[0, d] == bonus[0]


def test_tree_duplicate_siblings_take_lowest_index():
    parent = np.array([-1, 0, 0, 1, 2])
    tok = np.array([[0, 4, 4, 1, 2]])
    logits = np.zeros((1, 5, 6))
    logits[0, 0, 4] = 1      # root predicts 4: nodes 1 and 2 both match
    logits[0, 1, 5] = 1      # node 1 predicts 5 (its child 3 has token 1: no match)
    logits[0, 2, 2] = 1      # node 2 predicts 2 (its child 4 would match)
    acc, path, com, bonus = A.accept_tree_greedy(logits, tok, parent)
    assert acc[0] == 1 and path[0, 0] == 1 and bonus[0] == 5


def test_chain_tree_equals_chain():
    rng = np.random.default_rng(8)
    for _ in range(100):
        W, V = 5, 4
        logits = rng.normal(size=(1, W, V))
        am = logits[0].argmax(-1)
        x = np.where(rng.random(W - 1) < 0.7, am[:-1], rng.integers(0, V, W - 1))
        tok = np.concatenate([[0], x])[None]
        acc_t, _, com_t, _ = A.accept_tree_greedy(logits, tok, np.arange(-1, W - 1))
        acc_c, com_c, _ = A.accept_greedy(logits, x[None])
        assert acc_t[0] == acc_c[0]
        np.testing.assert_array_equal(com_t[0], com_c[0])


def test_tree_counting_exercise9(golden):
    g = golden("tree_exercise9.json")
    assert M.tree_nodes(g["branching"]) == g["draft_tokens"]
    e = M.tree_expected_accepts(g["topk_hit_per_level"])
    assert abs(e - g["expected_accepted"]) <= 0.005
    assert abs(1 + e - g["tau"]) <= 0.005
    # the 15-node verify tree: binary branching, three levels below the root
    assert 1 + M.tree_nodes([2, 2, 2]) == 15
