"""Acceptance rules of one verify round (oracle; test infrastructure only).

Layout of one round for sequence b (verify block, window width W = gamma + 1):
row 0 holds the pending token (the last committed token, whose KV is not yet in
the cache), rows 1..gamma hold the drafts x_1..x_gamma.  Row j's logits give the
target distribution of the token after row j, so the draft x_i is tested
against row i-1, and row gamma is the bonus distribution.

Sources:
* Greedy: "Per-step cost versus accepted tokens", section "What SGLang actually
  runs" -- compare each draft with the target argmax at its position, take the
  cumulative product of the matches; its sum is the accepted length; the round
  commits the accepted drafts plus one target token.  Lecture 6 "Optimizing
  Autoregressive Decode" section 7.4 -- at temperature 0 the rule reduces to
  exactly this, and the output equals the target's own greedy decode.
* Stochastic: Lecture 6 section 6.2 (Leviathan Algorithm 1): accept x_i while a
  uniform r_i < p_i(x_i)/q_i(x_i), stop at the first rejection; after a
  rejection at position n+1 draw from norm(max(0, p_{n+1} - q_{n+1})); after
  full acceptance draw the bonus from p_{gamma+1}.  Section 7.1 proves the
  output law equals p; section 7.2 gives P(accept) = sum min(p, q) = 1 - TV.
* Tree: Lecture 6 section 10.3 -- one forward over a token tree under an
  ancestor mask; greedy acceptance keeps the longest root-to-leaf path whose
  tokens match the target argmax.

Readings where the pages leave a step open:
* The test r_i < p/q is evaluated as fl32(u * q(x)) < p(x): no division, the
  same set of outcomes for q > 0; q(x) = 0 < p(x) accepts, p(x) = 0 rejects.
* Uniforms u[b, 0..gamma-1] drive the tests, u[b, gamma] drives the one final
  draw (residual or bonus); exactly one final draw happens per round.
* The final draw is an integer inverse CDF (see `draw_index`) so that it is
  reproducible bit for bit under any summation order.
* Greedy ties go to the lowest token index.
* A final draw whose target row has no mass on the 2^-40 grid at all (an input
  that is not a distribution, e.g. an all-zero row given to the standalone
  acceptance; a softmax row always has mass) returns token 0, chain and tree alike.
* Sampling adjustments (`adjust_probs`): temperature first (in `target_probs`),
  then top-k, then top-p over the top-k renormalised distribution; rank order is
  p descending with the lower token index first on equal p; masses on the same
  2^-40 grid as the final draw, so set membership is exact integer arithmetic.
"""
from __future__ import annotations

import numpy as np

TWO_POW_40 = float(2 ** 40)
TWO_POW_24 = float(2 ** 24)
MASK24 = np.uint64((1 << 24) - 1)


# ----------------------------------------------------------------------------- p
def target_probs(logits: np.ndarray, temperature: float) -> np.ndarray:
    """p = softmax(logits / T) over the last axis, in float64, rounded to float32.

    Lecture 6 section 7.3: temperature sampling is sampling from softmax(logits/T).
    """
    z = np.asarray(logits, dtype=np.float64) / float(temperature)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


# ---------------------------------------------------------- sampling adjustments
def adjust_probs(p_row: np.ndarray, top_k: int, top_p: float) -> np.ndarray:
    """Top-k then top-p (nucleus) renormalisation of one probability row.

    Lecture 6 "Optimizing Autoregressive Decode" section 7.3: each sampling setting
    is sampling from an adjusted distribution (top-k: every token ranked after the
    k-th gets probability zero; top-p: the smallest set of top-ranked tokens whose
    mass reaches p), and speculative sampling on the adjusted p and q follows the
    adjusted p.  "Per-step cost versus accepted tokens", section "Reefs": the
    renormalisation after top-k / top-p happens at verify time, for top_p < 1 or
    top_k > 1.  Readings (the pages fix neither the order nor the arithmetic):

    * rank order: p descending, lower token index first among equal p;
    * top_k in [1, V) is active (0 or >= V: off); top_p in (0, 1) is active (1: off);
    * masses R_v = floor(p_v * 2^40) (the final draw's grid); with the first k ranked
      tokens (all V when top-k is off) of mass S_k, the nucleus is the shortest
      ranked prefix (at least one token) whose mass reaches
      ceil(fl64(top_p) * S_k) -- top-p acts on the top-k renormalised distribution;
    * kept tokens get fl32(fl64(R_v) * fl64(1 / Z)), Z = their summed mass (a
      float64 reciprocal, then one float64 product per token); all others 0.  With
      no adjustment active, or Z = 0, p is returned unchanged.
    """
    p = np.asarray(p_row, dtype=np.float32)
    V = p.size
    k_on = 1 <= int(top_k) < V
    p_on = float(np.float32(top_p)) < 1.0
    if not (k_on or p_on):
        return p.copy()
    pk = np.where(p > 0, p, np.float32(0.0))
    order = np.lexsort((np.arange(V), -pk.astype(np.float64)))   # last key is primary
    R = [int(r) for r in fixed_point_mass(pk[order])]
    n = int(top_k) if k_on else V
    if p_on:
        s_k = sum(R[:n])
        tau = max(1, int(np.ceil(np.float64(np.float32(top_p)) * np.float64(s_k))))
        run, n_p = 0, n
        for i in range(n):
            run += R[i]
            if run >= tau:
                n_p = i + 1
                break
        n = n_p
    Z = sum(R[:n])
    if Z == 0:
        return p.copy()
    out = np.zeros(V, dtype=np.float32)
    inv = np.float64(1.0) / np.float64(Z)
    out[order[:n]] = (np.array(R[:n], dtype=np.float64) * inv).astype(np.float32)
    return out


def adjust_rows(p: np.ndarray, top_k, top_p) -> np.ndarray:
    """`adjust_probs` on every row of p [B, W, V]; top_k, top_p per sequence [B]."""
    p = np.asarray(p, dtype=np.float32)
    out = np.empty_like(p)
    for b in range(p.shape[0]):
        for j in range(p.shape[1]):
            out[b, j] = adjust_probs(p[b, j], int(np.asarray(top_k)[b]), float(np.asarray(top_p)[b]))
    return out


# ------------------------------------------------------------------- greedy chain
def accept_greedy(logits: np.ndarray, x: np.ndarray):
    """Greedy longest-matching-prefix acceptance.

    logits [B, W, V] (any float), x [B, gamma] drafts.  Returns
    (accepted [B], committed [B, W] with -1 after the first n+1 entries, bonus [B]).
    """
    logits = np.asarray(logits)
    B, W, _ = logits.shape
    gamma = W - 1
    a = np.argmax(logits, axis=-1)                 # first maximal index on ties
    match = (np.asarray(x).reshape(B, gamma) == a[:, :gamma]).astype(np.int64)
    n = np.cumprod(match, axis=1).sum(axis=1) if gamma > 0 else np.zeros(B, np.int64)
    bonus = a[np.arange(B), n]
    committed = np.full((B, W), -1, dtype=np.int64)
    for b in range(B):
        committed[b, :n[b]] = x[b, :n[b]]
        committed[b, n[b]] = bonus[b]
    return n.astype(np.int64), committed, bonus.astype(np.int64)


# ----------------------------------------------------------------- stochastic chain
def accept_test(u: np.ndarray, q_x: np.ndarray, p_x: np.ndarray) -> np.ndarray:
    """r < p/q evaluated as fl32(u * q) < p (float32, no fused multiply-add)."""
    prod = np.multiply(np.float32(1.0) * u.astype(np.float32), q_x.astype(np.float32),
                       dtype=np.float32)
    return prod < p_x.astype(np.float32)


def residual(p_row: np.ndarray, q_row: np.ndarray) -> np.ndarray:
    """max(0, p - q) in float32 (unnormalised; the draw normalises)."""
    return np.maximum(np.float32(0.0), (p_row.astype(np.float32) - q_row.astype(np.float32)))


def fixed_point_mass(r: np.ndarray) -> np.ndarray:
    """R_v = floor(r_v * 2^40) as uint64.  Exact: r is float32 <= 1."""
    return np.floor(np.asarray(r, dtype=np.float32).astype(np.float64) * TWO_POW_40).astype(np.uint64)


def draw_index(R: np.ndarray, u: float) -> int:
    """Integer inverse-CDF draw from the unnormalised masses R (uint64, one row).

    S = sum R, m = floor(u * 2^24), t = floor(m * S / 2^24); return the smallest
    v with R_0 + ... + R_v > t.  P(v) = R_v / S up to the 2^-24 grid of u.
    Returns -1 when S == 0.  Written with Python integers (no overflow).
    """
    S = int(np.sum(R, dtype=np.uint64))
    if S == 0:
        return -1
    m = int(np.floor(np.float64(np.float32(u)) * TWO_POW_24))
    t = (m * S) >> 24
    c = np.cumsum(R, dtype=np.uint64)
    return int(np.searchsorted(c, np.uint64(t), side="right"))


def draw_index_rows(R: np.ndarray, u: np.ndarray) -> np.ndarray:
    """`draw_index` for many rows at once: R [B, V] uint64, u [B] float32.

    (m * S) >> 24 is formed without a 128-bit product through the identity
    m*S = m*S_hi*2^24 + m*S_lo with S_hi = S >> 24, S_lo = S mod 2^24, so
    (m*S) >> 24 = m*S_hi + ((m*S_lo) >> 24); both terms fit in 64 bits
    because m < 2^24 and S < 2^58.
    """
    R = np.asarray(R, dtype=np.uint64)
    S = R.sum(axis=1, dtype=np.uint64)
    m = np.floor(np.asarray(u, dtype=np.float32).astype(np.float64) * TWO_POW_24).astype(np.uint64)
    t = m * (S >> np.uint64(24)) + ((m * (S & MASK24)) >> np.uint64(24))
    c = np.cumsum(R, axis=1, dtype=np.uint64)
    idx = (c <= t[:, None]).sum(axis=1).astype(np.int64)
    idx[S == 0] = -1
    return idx


def accept_stochastic(p: np.ndarray, q: np.ndarray, x: np.ndarray, u: np.ndarray,
                      accept_fn=accept_test, residual_fn=residual):
    """Chain rejection sampling (Leviathan Algorithm 1) for a batch of rounds.

    p [B, W, V] float32 target probabilities (row j = p_{j+1}), q [B, gamma, V]
    float32 draft probabilities (q[:, i-1] = q_i), x [B, gamma] drafts, u [B, W]
    float32 uniforms.  gamma = 0 is a plain sample from p (the decode step).

    Returns (accepted [B], committed [B, W] (-1 padded), final [B], zero_residual [B])
    where zero_residual flags rounds whose residual had no mass on the 2^-40 grid;
    those draw from p at the break row instead.  A row of p with no mass on the
    grid either (all zeros: not a distribution, so never a softmax row) gives
    token 0.
    """
    p = np.asarray(p, dtype=np.float32)
    B, W, V = p.shape
    gamma = W - 1
    x = np.asarray(x, dtype=np.int64).reshape(B, gamma)
    u = np.asarray(u, dtype=np.float32).reshape(B, W)
    bi = np.arange(B)
    n = np.zeros(B, dtype=np.int64)
    alive = np.ones(B, dtype=bool)
    for i in range(gamma):
        xi = x[:, i]
        ok = accept_fn(u[:, i], q[bi, i, xi], p[bi, i, xi])
        alive &= ok
        n += alive
    rejected = n < gamma
    r = p[bi, n].copy()                          # full acceptance: bonus from p_{gamma+1}
    if gamma > 0 and rejected.any():
        rb = bi[rejected]
        r[rb] = residual_fn(p[rb, n[rb]], q[rb, n[rb]])
    R = fixed_point_mass(r)
    tok = draw_index_rows(R, u[:, gamma])
    zero = tok < 0
    if zero.any():
        tok[zero] = draw_index_rows(fixed_point_mass(p[bi[zero], n[zero]]), u[zero, gamma])
    tok[tok < 0] = 0                             # p without mass: token 0
    committed = np.full((B, W), -1, dtype=np.int64)
    for b in range(B):
        committed[b, :n[b]] = x[b, :n[b]]
        committed[b, n[b]] = tok[b]
    return n, committed, tok, zero


def accept_stochastic_from_logits(logits, q, x, u, temperature: float):
    """The verify round's acceptance as the library runs it: p from the logits, then
    `accept_stochastic`.  Also returns the margins of each decision."""
    p = target_probs(logits, temperature)
    return accept_stochastic(p, q, x, u), p


# --------------------------------------------------------------------------- tree
def tree_depths(parent: np.ndarray) -> np.ndarray:
    """Depth of every node; parent[0] = -1 (root), parent[c] < c (BFS order)."""
    parent = np.asarray(parent, dtype=np.int64)
    depth = np.zeros(len(parent), dtype=np.int64)
    for c in range(1, len(parent)):
        assert 0 <= parent[c] < c, "nodes must be in BFS order with parent < child"
        depth[c] = depth[parent[c]] + 1
    return depth


def tree_ancestors(parent: np.ndarray) -> list:
    """For each node, the set of its ancestors including itself."""
    parent = np.asarray(parent, dtype=np.int64)
    anc = []
    for c in range(len(parent)):
        s = {c}
        v = c
        while parent[v] >= 0:
            v = int(parent[v])
            s.add(v)
        anc.append(s)
    return anc


def accept_tree_greedy(logits: np.ndarray, tok: np.ndarray, parent: np.ndarray):
    """Greedy walk of a token tree: from the root, move to the child whose token is
    the target argmax at the current node (lowest node index if several), stop when
    none matches; the argmax at the stopping node is the bonus token.

    logits [B, N, V], tok [B, N] (node 0 = pending token), parent [N].
    Returns (accepted [B], path [B, maxdepth] node ids (-1 padded),
             committed [B, maxdepth+1] tokens (-1 padded), bonus [B]).
    """
    logits = np.asarray(logits)
    B, N, _ = logits.shape
    parent = np.asarray(parent, dtype=np.int64)
    depth = tree_depths(parent)
    dmax = int(depth.max())
    accepted = np.zeros(B, dtype=np.int64)
    path = np.full((B, max(dmax, 1)), -1, dtype=np.int64)
    committed = np.full((B, dmax + 1), -1, dtype=np.int64)
    bonus = np.zeros(B, dtype=np.int64)
    for b in range(B):
        v, k = 0, 0
        while True:
            a = int(np.argmax(logits[b, v]))
            nxt = -1
            for c in range(1, N):
                if parent[c] == v and int(tok[b, c]) == a:
                    nxt = c
                    break
            if nxt < 0:
                break
            path[b, k] = nxt
            committed[b, k] = a
            k += 1
            v = nxt
        accepted[b] = k
        committed[b, k] = a
        bonus[b] = a
    return accepted, path, committed, bonus


# ------------------------------------------------------------------ stochastic tree
def residual_step(p_cur: np.ndarray, q_row: np.ndarray):
    """One rejection of recursive rejection sampling over sibling candidates:
    r = max(0, p - q) in float32, masses R = floor(r * 2^40), Z = sum R (exact), and
    the normalised residual fl32(fl64(R) * fl64(1/Z)).  Z == 0 (no residual mass on
    the grid, which exact arithmetic never reaches after a rejection) keeps p."""
    r = residual(p_cur, q_row)
    R = fixed_point_mass(r)
    Z = int(np.sum(R, dtype=np.uint64))
    if Z == 0:
        return np.asarray(p_cur, np.float32).copy(), R
    inv = np.float64(1.0) / np.float64(Z)
    return (R.astype(np.float64) * inv).astype(np.float32), R


def accept_tree_stochastic(p: np.ndarray, q, tok: np.ndarray, parent: np.ndarray, u: np.ndarray):
    """Stochastic verification of a token tree (multi-draft speculative sampling).

    Lecture 6 "Optimizing Autoregressive Decode" section 10.3: a tree of candidates
    (SpecInfer, Miao et al. 2024) is verified in one forward under an ancestor mask;
    "Per-step cost versus accepted tokens", section "Reefs": sampled (non-greedy)
    tree verification exists beside the chain sampler.  The pages leave the rule
    open; this is SpecInfer's multi-step speculative sampling, i.e. recursive
    rejection sampling over the children of a node:

    * at node v the target is p_cur = p[v]; the children c of v are tried in node
      order: child c (token x) is accepted when fl32(u[c] * q_v(x)) < p_cur(x), and
      the walk moves to c;
    * after a rejection p_cur becomes the normalised residual max(0, p_cur - q_v)
      (`residual_step`); after the last child is rejected the final token is drawn
      from that residual (unnormalised masses, integer inverse CDF, u[0]);
    * at a node without children the final (bonus) token is drawn from p[v] (u[0]).

    q[b, v] is the distribution the children of node v were drawn from (i.i.d.);
    q = None means deterministic candidates ("target only"): each child's q is the
    one-hot of its own token, so a child is accepted with probability p_cur(x) and
    a rejection removes x from the target.  With one child per node this is the
    chain rule of `accept_stochastic` (tree u[c] = chain u[c-1], tree u[0] = chain
    u[gamma]).

    p [B, N, V] float32 (row c = target after node c), q [B, N, V] or None,
    tok [B, N] (node 0 = pending token), parent [N] (BFS order), u [B, N] float32.
    Returns (accepted [B], path [B, maxdepth] node ids (-1 padded),
             committed [B, maxdepth+1] tokens (-1 padded), final [B]).
    """
    p = np.asarray(p, dtype=np.float32)
    B, N, V = p.shape
    parent = np.asarray(parent, dtype=np.int64)
    depth = tree_depths(parent)
    dmax = int(depth.max())
    u = np.asarray(u, dtype=np.float32).reshape(B, N)
    children = [[c for c in range(1, N) if parent[c] == v] for v in range(N)]
    accepted = np.zeros(B, dtype=np.int64)
    path = np.full((B, max(dmax, 1)), -1, dtype=np.int64)
    committed = np.full((B, dmax + 1), -1, dtype=np.int64)
    final = np.zeros(B, dtype=np.int64)
    for b in range(B):
        v, k = 0, 0
        while True:
            p_cur = p[b, v]
            moved, R_last = -1, None
            for j, c in enumerate(children[v]):
                x = int(tok[b, c])
                if q is None:
                    q_row = np.zeros(V, np.float32)
                    q_row[x] = 1.0
                else:
                    q_row = np.asarray(q[b, v], np.float32)
                if accept_test(u[b, c:c + 1], q_row[x:x + 1], p_cur[x:x + 1])[0]:
                    moved = c
                    break
                p_next, R_last = residual_step(p_cur, q_row)
                if j == len(children[v]) - 1:
                    break
                p_cur = p_next
            if moved >= 0:
                path[b, k] = moved
                committed[b, k] = int(tok[b, moved])
                k += 1
                v = moved
                continue
            if R_last is None:                       # no children: bonus from p at v
                R_last = fixed_point_mass(p[b, v])
            t = draw_index(R_last, float(u[b, 0]))
            if t < 0:                                # residual without mass: draw from p_cur
                t = draw_index(fixed_point_mass(p_cur), float(u[b, 0]))
            if t < 0:                                # no mass at all (not a distribution): token 0
                t = 0
            final[b] = t
            committed[b, k] = t
            accepted[b] = k
            break
    return accepted, path, committed, final
