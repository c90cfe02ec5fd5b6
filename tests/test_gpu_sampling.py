"""Top-k / top-p sampling adjustments on the GPU against the oracle.

Standalone (identical probabilities in): the adjusted rows, and acceptance on
adjusted p and q, are bit-exact.  Model rounds (logits from the tiny decoder):
bit-exact wherever the oracle's decisions, including the kept sets, are clear of
the margins; top_k = 1 turns a sampled round into the greedy round exactly."""
import numpy as np
import pytest
import torch

from oracle import accept as A
from speculative_decoding_verify_step_gb300 import synth
from tests._gpu import cuda_model, need_gpu, oracle_for, stochastic_margin

pytestmark = pytest.mark.gpu


def _spec():
    from speculative_decoding_verify_step_gb300 import spec
    return spec


def _rows(kind, n, V, seed):
    g = np.random.default_rng(seed)
    if kind == "dirichlet":
        return g.dirichlet(np.full(V, 0.3), size=n).astype(np.float32)
    if kind == "softmax":
        z = g.normal(size=(n, V)) * g.uniform(1, 8, size=(n, 1))
        e = np.exp(z - z.max(-1, keepdims=True))
        return (e / e.sum(-1, keepdims=True)).astype(np.float32)
    if kind == "ties":        # exact ties: multiples of 2^-18 (sum < 1)
        c = g.integers(0, 4, size=(n, V)).astype(np.float64)
        c *= min(1.0, 0.9 * 2 ** 18 / c.sum(-1).max())
        return (np.floor(c) / 2 ** 18).astype(np.float32)
    if kind == "uniform":
        return np.full((n, V), 1.0 / V, np.float32)
    raise ValueError(kind)


SETTINGS = [(0, 1.0), (1, 1.0), (2, 1.0), (50, 1.0), (-2, 1.0), (0, 0.5), (0, 0.9), (0, 0.95), (0, 1e-6),
            (50, 0.9), (3, 0.3), (0, 1.5), (7, 0.999)]


@pytest.mark.parametrize("V", [1000, 1024, 50257, 128256])
@pytest.mark.parametrize("kind", ["dirichlet", "softmax", "ties", "uniform"])
def test_adjust_probs_bit_exact(V, kind):
    need_gpu()
    spec = _spec()
    per = 2                                     # rows per setting
    settings = SETTINGS + [(V - 1, 1.0), (V, 1.0), (V // 2, 0.7)]
    n = per * len(settings)
    p = _rows(kind, n, V, seed=V + len(kind))
    k = np.array([s[0] for s in settings], np.int32)
    tp = np.array([s[1] for s in settings], np.float32)
    got = spec.spec_adjust_probs(torch.from_numpy(p).cuda(), top_k=k, top_p=tp, rows_per_setting=per).cpu().numpy()
    for r in range(n):
        kk, pp = int(k[r // per]), float(tp[r // per])
        bad = kk < 0 or not (0 < pp <= 1)
        want = p[r] if bad else A.adjust_probs(p[r], kk, pp)
        np.testing.assert_array_equal(got[r].view(np.int32), want.view(np.int32), err_msg=f"row {r} k={kk} p={pp}")


def test_adjust_probs_in_place_and_null_settings():
    need_gpu()
    spec = _spec()
    p = torch.from_numpy(_rows("softmax", 3, 5000, 1)).cuda()
    ref = p.clone()
    same = spec.spec_adjust_probs(p)             # both settings NULL: a copy
    assert torch.equal(same, ref)
    spec.spec_adjust_probs(p, top_k=[5], rows_per_setting=3, out=p)
    want = np.stack([A.adjust_probs(r, 5, 1.0) for r in ref.cpu().numpy()])
    np.testing.assert_array_equal(p.cpu().numpy(), want)


@pytest.mark.parametrize("V", [1024, 128256])
def test_acceptance_on_adjusted_rows_bit_exact(V):
    """p and q adjusted alike (per sequence), then the standalone acceptance."""
    need_gpu()
    spec = _spec()
    B, gamma = 6, 3
    W = gamma + 1
    g = np.random.default_rng(V)
    p = _rows("softmax", B * W, V, seed=3).reshape(B, W, V)
    q = (0.5 * p[:, :gamma] + 0.5 * _rows("dirichlet", B * gamma, V, seed=4).reshape(B, gamma, V)).astype(np.float32)
    k = np.array([0, 1, 5, 40, 0, 3], np.int32)
    tp = np.array([0.9, 1.0, 1.0, 0.8, 0.5, 0.95], np.float32)
    pa, qa = A.adjust_rows(p, k, tp), A.adjust_rows(q, k, tp)
    x = np.zeros((B, gamma), np.int64)
    for b in range(B):
        for i in range(gamma):
            c = np.cumsum(qa[b, i].astype(np.float64))
            x[b, i] = min(int(np.searchsorted(c, g.random() * c[-1], side="right")), V - 1)
    u = g.random((B, W)).astype(np.float32)
    n_ref, com_ref, tok_ref, _ = A.accept_stochastic(pa, qa, x, u)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    pa_g = spec.spec_adjust_probs(d(p), top_k=k, top_p=tp, rows_per_setting=W)
    qa_g = spec.spec_adjust_probs(d(q), top_k=k, top_p=tp, rows_per_setting=gamma)
    np.testing.assert_array_equal(pa_g.cpu().numpy(), pa)
    np.testing.assert_array_equal(qa_g.cpu().numpy(), qa)
    acc, com, bon = spec.spec_accept_probs(pa_g, qa_g, d(x), d(u))
    np.testing.assert_array_equal(acc.cpu().numpy(), n_ref)
    np.testing.assert_array_equal(com.cpu().numpy(), com_ref)
    np.testing.assert_array_equal(bon.cpu().numpy(), tok_ref)


# ------------------------------------------------------------------ model rounds
KW = dict(max_batch=4, max_width=8, max_seq_len=512, num_pages=40)
SHARP = 8.0   # final-norm gain factor: logits of std ~2.5 instead of ~0.3 (peaked rows)


@pytest.fixture(scope="module")
def sharp_tiny():
    need_gpu()
    w = synth.make_weights(synth.TINY, seed=4, gain_jitter=0.1)
    w["final_norm"] = w["final_norm"] * SHARP
    m = cuda_model(synth.TINY, w, **KW)
    yield w, m
    m.close()


def _fresh(w, m, prompts, with_oracle=True):
    ids = list(range(len(prompts)))
    m.seq_reset(ids)
    L = max(len(p) for p in prompts)
    tok = torch.zeros(len(prompts), L, dtype=torch.int32)
    for b, p in enumerate(prompts):
        tok[b, :len(p)] = torch.as_tensor(p)
    m.prefill(ids, tok.cuda(), [len(p) for p in prompts])
    if not with_oracle:
        return ids, None
    o = oracle_for(synth.TINY, w, **KW)
    o.prefill(ids, prompts)
    return ids, o


def set_clear(p_row, k, tp, margin=1e-2):
    """The kept set of `adjust_probs` is fixed by the reference row when the last kept
    and the first dropped token (at the top-k and at the nucleus boundary) differ by
    more than the margin relative, and the nucleus threshold sits more than margin x
    itself from the cumulative mass on both sides."""
    V = p_row.size
    k_on, p_on = 1 <= k < V, tp < 1
    s = np.sort(p_row.astype(np.float64))[::-1]
    n = k if k_on else V
    if k_on and s[k - 1] <= (1 + margin) * s[k]:
        return False
    if p_on:
        c = np.cumsum(s[:n])
        tau = tp * c[-1]
        j = int(np.searchsorted(c, tau, side="left"))       # first prefix reaching tau
        if c[j] < (1 + margin) * tau or (j > 0 and c[j - 1] > (1 - margin) * tau):
            return False
        if j + 1 < V and s[j] <= (1 + margin) * s[j + 1]:
            return False
    return True


@pytest.mark.parametrize("k,tp", [(3, 1.0), (0, 0.3), (6, 0.5)])
def test_sampled_rounds_with_adjustments(sharp_tiny, k, tp):
    """Settings whose kept sets are mostly clear of the margins on these peaked rows
    (a nucleus boundary is clear only when the crossing token moves the cumulative
    mass well past the threshold, so small top_p values are the informative ones)."""
    w, m = sharp_tiny
    V, gamma, B = synth.TINY.vocab, 2, 4
    compared = 0
    for seed in range(8):
        g = np.random.default_rng(100 * seed + k)
        prompts = [g.integers(0, V, n) for n in (40, 66, 90, 51)]
        ids, o = _fresh(w, m, prompts)
        # drafts from the adjusted mixture of the oracle's target and Dir(1)
        tok = np.zeros((B, gamma + 1), np.int64)
        tok[:, 0] = [p_[-1] for p_ in prompts]
        q = np.zeros((B, gamma, V), np.float32)
        D = synth.dirichlet1((B, gamma, V), seed=seed).numpy()
        for i in range(gamma):
            pi = A.target_probs(o.forward(ids, tok[:, :i + 1])[:, i], 1.0)
            for b in range(B):
                q[b, i] = A.adjust_probs((0.6 * pi[b] + 0.4 * D[b, i]).astype(np.float32), k, tp)
                c = np.cumsum(q[b, i].astype(np.float64))
                tok[b, i + 1] = min(int(np.searchsorted(c, g.random() * c[-1], side="right")), V - 1)
        u = synth.uniforms((B, gamma + 1), seed=50 + seed).numpy()
        logits = o.forward(ids, tok)
        p = A.target_probs(logits, 1.0)
        pa = A.adjust_rows(p, [k] * B, [tp] * B)
        n_ref, com_ref, _, _ = A.accept_stochastic(pa, q, tok[:, 1:], u)
        clear = stochastic_margin(pa, q, tok[:, 1:], u, n_ref)
        for b in range(B):
            clear[b] &= all(set_clear(p[b, j], k, tp) for j in range(int(n_ref[b]) + 1))
        acc, com, _ = m.verify_step(ids, torch.from_numpy(tok).cuda(), q=torch.from_numpy(q).cuda(),
                                    u=torch.from_numpy(u).cuda(), temperature=1.0, top_k=[k] * B, top_p=[tp] * B)
        m.sync_status()
        acc, com = acc.cpu().numpy(), com.cpu().numpy()
        for b in range(B):
            if clear[b]:
                compared += 1
                assert acc[b] == n_ref[b], (seed, b)
                np.testing.assert_array_equal(com[b], com_ref[b])
    assert compared >= 8, compared


def _round_inputs(m, B, gamma, seed):
    V = synth.TINY.vocab
    g = np.random.default_rng(seed)
    prompts = [g.integers(0, V, n) for n in (50, 70, 33, 64)[:B]]
    return prompts, g


def test_top1_sampled_verify_is_greedy_verify(sharp_tiny):
    """top_k = 1: every adjusted row is the argmax one-hot, so the sampled round takes
    exactly the greedy round's decisions, whatever q and u are."""
    w, m = sharp_tiny
    V, gamma, B = synth.TINY.vocab, 4, 4
    for seed in range(3):
        prompts, g = _round_inputs(m, B, gamma, seed)
        tok = np.concatenate([np.array([[p_[-1]] for p_ in prompts]), g.integers(0, V, (B, gamma))], axis=1)
        ids, _ = _fresh(w, m, prompts, False)
        lg = m.score(ids, torch.from_numpy(tok).cuda()).cpu().numpy()
        am = lg.argmax(-1)
        tok[:, 1:3] = am[:, 0:2]                     # the first drafts are the argmax: some acceptance
        q = torch.from_numpy(synth.dirichlet1((B, gamma, V), seed=seed).numpy()).cuda()
        u = torch.from_numpy(g.random((B, gamma + 1)).astype(np.float32)).cuda()
        t = torch.from_numpy(tok).cuda()
        ids, _ = _fresh(w, m, prompts, False)
        a1, c1, b1 = m.verify_step(ids, t, q=q, u=u, temperature=1.0, top_k=[1] * B)
        ids, _ = _fresh(w, m, prompts, False)
        a2, c2, b2 = m.verify_step(ids, t)
        assert torch.equal(a1, a2) and torch.equal(c1, c2) and torch.equal(b1, b2)
        # the same through a vanishing nucleus, the ragged compact round and the decode step
        ids, _ = _fresh(w, m, prompts, False)
        a3, c3, _ = m.verify_step(ids, t, q=q, u=u, temperature=0.7, top_p=[1e-7] * B)
        assert torch.equal(a3, a2) and torch.equal(c3, c2)
        lens = [5, 3, 1, 4]
        packed = torch.cat([t[b, :lens[b]] for b in range(B)])
        spec = _spec()
        ids, _ = _fresh(w, m, prompts, False)
        a4, c4, _ = m.verify_ragged(ids, packed, lens, spec.RAGGED_COMPACT, q=q, u=u, temperature=1.0, gamma=gamma,
                                    top_k=[1] * B)
        ids, _ = _fresh(w, m, prompts, False)
        a5, c5, _ = m.verify_ragged(ids, packed, lens, spec.RAGGED_COMPACT, gamma=gamma)
        assert torch.equal(a4, a5) and torch.equal(c4, c5)
        ids, _ = _fresh(w, m, prompts, False)
        d1 = m.decode_step(ids, t[:, 0], temperature=1.0, u=u[:, 0].contiguous(), top_k=[1] * B)
        ids, _ = _fresh(w, m, prompts, False)
        d2 = m.decode_step(ids, t[:, 0])
        assert torch.equal(d1, d2)
        m.sync_status()


def test_bad_setting_is_reported(sharp_tiny):
    w, m = sharp_tiny
    spec = _spec()
    prompts, g = _round_inputs(m, 2, 2, 7)
    ids, _ = _fresh(w, m, prompts, False)
    tok = torch.from_numpy(g.integers(0, synth.TINY.vocab, (2, 3))).int().cuda()
    q = torch.from_numpy(synth.dirichlet1((2, 2, synth.TINY.vocab), seed=1).numpy()).cuda()
    u = torch.full((2, 3), 0.5, device="cuda")
    m.verify_step(ids, tok, q=q, u=u, temperature=1.0, top_k=[3, -1])
    with pytest.raises(spec.SpecError) as e:
        m.sync_status()
    assert e.value.status == 1
