"""Sampled token-tree verification on the GPU against the oracle.

Standalone (identical probabilities in): accepted counts, committed tokens and
final tokens are bit-exact for i.i.d. and deterministic candidates, chains, stars
and binary trees, up to the full 8B vocabulary.  Model rounds (tiny decoder): the
same decisions wherever the oracle's are stable under a 1% perturbation of the
target rows, and the path's KV compaction and page tables follow the oracle."""
import numpy as np
import pytest
import torch

from oracle import accept as A
from speculative_decoding_verify_step_gb300 import synth
from tests._gpu import cuda_model, need_gpu, oracle_for, rel_err

pytestmark = pytest.mark.gpu

TREES = {
    "chain5": [-1, 0, 1, 2, 3],
    "star4": [-1, 0, 0, 0, 0],
    "binary7": [-1, 0, 0, 1, 1, 2, 2],
    "binary15": [-1, 0, 0, 1, 1, 2, 2, 3, 3, 4, 4, 5, 5, 6, 6],
    "mixed9": [-1, 0, 0, 0, 1, 1, 3, 6, 6],
}


def _spec():
    from speculative_decoding_verify_step_gb300 import spec
    return spec


def _draw(g, row):
    c = np.cumsum(row.astype(np.float64))
    return min(int(np.searchsorted(c, g.random() * c[-1], side="right")), len(row) - 1)


def _inputs(B, parent, V, iid, seed):
    """Target rows, draft rows, candidate tokens (drawn from q, or distinct top tokens
    of q for deterministic candidates) and uniforms."""
    g = np.random.default_rng(seed)
    N = len(parent)
    z = g.normal(size=(B, N, V)) * g.uniform(1, 4, size=(B, N, 1))
    p = np.exp(z - z.max(-1, keepdims=True))
    p = (p / p.sum(-1, keepdims=True)).astype(np.float32)
    q = (0.5 * p + 0.5 * g.dirichlet(np.full(V, 0.5), size=(B, N))).astype(np.float32)
    tok = np.zeros((B, N), np.int64)
    for b in range(B):
        for v in range(N):
            kids = [c for c in range(1, N) if parent[c] == v]
            if iid:
                for c in kids:
                    tok[b, c] = _draw(g, q[b, v])
            else:
                top = np.argsort(-q[b, v], kind="stable")[:len(kids)]
                for c, t in zip(kids, top):
                    tok[b, c] = t
    u = g.random((B, N)).astype(np.float32)
    return p, q, tok, u


@pytest.mark.parametrize("V", [40, 1024, 128256])
@pytest.mark.parametrize("tree", list(TREES))
@pytest.mark.parametrize("iid", [True, False])
def test_standalone_bit_exact(V, tree, iid):
    need_gpu()
    spec = _spec()
    parent = TREES[tree]
    B = 6 if V < 100000 else 3
    for seed in range(3 if V < 100000 else 1):
        p, q, tok, u = _inputs(B, parent, V, iid, seed * 7 + len(tree) + V % 97)
        n_ref, path, com_ref, fin_ref = A.accept_tree_stochastic(p, q if iid else None, tok, np.array(parent), u)
        d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        acc, com, bon = spec.spec_accept_tree_probs(d(p), d(q) if iid else None, d(tok), parent, d(u))
        acc, com, bon = acc.cpu().numpy(), com.cpu().numpy(), bon.cpu().numpy()
        np.testing.assert_array_equal(acc, n_ref)
        np.testing.assert_array_equal(bon, fin_ref)
        dmax = com_ref.shape[1]
        np.testing.assert_array_equal(com[:, :dmax], com_ref)
        assert (com[:, dmax:] == -1).all()


def test_standalone_massless_rows_give_token_0():
    """Target rows without mass on the 2^-40 grid draw token 0, as in the oracle."""
    need_gpu()
    spec = _spec()
    parent = TREES["binary7"]
    for V in (1024, 128256):
        for iid in (True, False):
            p, q, tok, u = _inputs(4, parent, V, iid, seed=91)
            p[0] = 0.0
            p[1, 1:] = np.float32(2.0 ** -42)
            p[2, 0] = 0.0
            n_ref, path, com_ref, fin_ref = A.accept_tree_stochastic(p, q if iid else None, tok, np.array(parent), u)
            d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
            acc, com, bon = spec.spec_accept_tree_probs(d(p), d(q) if iid else None, d(tok), parent, d(u))
            np.testing.assert_array_equal(acc.cpu().numpy(), n_ref)
            np.testing.assert_array_equal(bon.cpu().numpy(), fin_ref)
            np.testing.assert_array_equal(com.cpu().numpy()[:, :com_ref.shape[1]], com_ref)
            assert fin_ref[0] == 0


def test_chain_tree_equals_chain_acceptance():
    """parent[c] = c - 1: the tree kernel takes the chain kernel's decisions."""
    need_gpu()
    spec = _spec()
    g = np.random.default_rng(3)
    B, gamma, V = 8, 5, 5000
    p = g.dirichlet(np.full(V, 0.3), size=(B, gamma + 1)).astype(np.float32)
    q = (0.5 * p[:, :gamma] + 0.5 * g.dirichlet(np.full(V, 0.3), size=(B, gamma))).astype(np.float32)
    x = np.array([[_draw(g, q[b, i]) for i in range(gamma)] for b in range(B)])
    u = g.random((B, gamma + 1)).astype(np.float32)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    a1, c1, b1 = spec.spec_accept_probs(d(p), d(q), d(x), d(u))
    tok = np.concatenate([np.zeros((B, 1), np.int64), x], 1)
    qt = np.concatenate([q, np.zeros((B, 1, V), np.float32)], 1)
    ut = np.concatenate([u[:, -1:], u[:, :-1]], 1)
    a2, c2, b2 = spec.spec_accept_tree_probs(d(p), d(qt), d(tok), list(range(-1, gamma)), d(ut))
    assert torch.equal(a1, a2) and torch.equal(b1, b2) and torch.equal(c1, c2)


# ------------------------------------------------------------------ model rounds
KW = dict(max_batch=4, max_width=16, max_seq_len=512, num_pages=40)
TREE = TREES["binary15"]


@pytest.fixture(scope="module")
def sharp_tiny():
    need_gpu()
    w = synth.make_weights(synth.TINY, seed=4, gain_jitter=0.1)
    w["final_norm"] = w["final_norm"] * 6.0       # peaked target rows
    m = cuda_model(synth.TINY, w, **KW)
    yield w, m
    m.close()


def _stable(p, q, tok, u, parent, n_ref, com_ref, trials=6, eps=1e-2, seed=0):
    """The oracle's decisions survive multiplicative 1% perturbations of the target
    rows (the GPU's rows differ from the oracle's by ~0.1%)."""
    g = np.random.default_rng(seed)
    B = p.shape[0]
    ok = np.ones(B, bool)
    for _ in range(trials):
        pp = p.astype(np.float64) * np.exp(eps * g.standard_normal(p.shape))
        pp = (pp / pp.sum(-1, keepdims=True)).astype(np.float32)
        n2, _, c2, _ = A.accept_tree_stochastic(pp, q, tok, np.array(parent), u)
        ok &= (n2 == n_ref) & (c2 == com_ref).all(axis=1)
    return ok


@pytest.mark.parametrize("iid", [True, False])
def test_model_rounds_match_oracle(sharp_tiny, iid):
    w, m = sharp_tiny
    V, N, B = synth.TINY.vocab, len(TREE), 3
    compared = 0
    for seed in range(6):
        g = np.random.default_rng(40 + seed + 10 * iid)
        prompts = [g.integers(0, V, n) for n in (50, 81, 66)]
        ids = list(range(B))
        m.seq_reset(ids)
        pt = torch.zeros(B, 81, dtype=torch.int32)
        for b, pr in enumerate(prompts):
            pt[b, :len(pr)] = torch.as_tensor(pr)
        m.prefill(ids, pt.cuda(), [len(pr) for pr in prompts])
        o = oracle_for(synth.TINY, w, **KW)
        o.prefill(ids, prompts)
        # candidates: drawn level by level from q = mixture of the oracle's target and Dir(1)
        tok = np.zeros((B, N), np.int64)
        tok[:, 0] = [pr[-1] for pr in prompts]
        q = np.zeros((B, N, V), np.float32)
        D = synth.dirichlet1((B, N, V), seed=seed).numpy()
        for v in range(N):
            kids = [c for c in range(1, N) if TREE[c] == v]
            if not kids:
                continue
            pv = A.target_probs(o.forward(ids, tok, parent=np.array(TREE))[:, v], 1.0)
            for b in range(B):
                q[b, v] = (0.6 * pv[b] + 0.4 * D[b, v]).astype(np.float32)
                if iid:
                    for c in kids:
                        tok[b, c] = _draw(g, q[b, v])
                else:
                    for c, t in zip(kids, np.argsort(-q[b, v], kind="stable")[:len(kids)]):
                        tok[b, c] = t
        u = g.random((B, N)).astype(np.float32)
        logits = o.forward(ids, tok, parent=np.array(TREE))
        p = A.target_probs(logits, 1.0)
        qq = q if iid else None
        n_ref, path, com_ref, fin_ref = A.accept_tree_stochastic(p, qq, tok, np.array(TREE), u)
        clear = _stable(p, qq, tok, u, TREE, n_ref, com_ref, seed=seed)
        L0 = o.lengths(ids)
        acc, com, bon = m.verify_tree_sampled(ids, torch.from_numpy(tok).cuda(), TREE, torch.from_numpy(u).cuda(),
                                              q=torch.from_numpy(q).cuda() if iid else None, temperature=1.0)
        m.sync_status()
        got = m.debug_logits(B * N).cpu().numpy().reshape(logits.shape)
        assert rel_err(got, logits) < 1e-2
        acc, com = acc.cpu().numpy(), com.cpu().numpy()
        dmax = com_ref.shape[1]
        for b in range(B):
            if clear[b]:
                compared += 1
                assert acc[b] == n_ref[b], (seed, b)
                np.testing.assert_array_equal(com[b, :dmax], com_ref[b])
        if clear.all():
            o.commit_tree(ids, path)
            lens, pt_ = m.kv_state(ids)
            assert lens == o.lengths(ids).tolist()
            np.testing.assert_array_equal(np.array(pt_), o.kv.page_table_array(ids))
            for b, s in enumerate(ids):          # compacted path KV, last layer
                layer = synth.TINY.n_layers - 1
                k, vv = m.read_kv(layer, s, int(L0[b]), int(n_ref[b]) + 1)
                kr = np.stack([o.kv.k[layer, o.kv.slot(s, t)[0], :, o.kv.slot(s, t)[1]]
                               for t in range(int(L0[b]), int(L0[b]) + int(n_ref[b]) + 1)])
                assert rel_err(k.float().numpy(), kr) < 1e-2
    assert compared >= 6, compared


def test_top1_sampled_tree_is_greedy_tree(sharp_tiny):
    """top_k = 1 with deterministic candidates: every target row is the argmax
    one-hot, so the sampled tree walk is the greedy walk."""
    w, m = sharp_tiny
    V, N, B = synth.TINY.vocab, len(TREE), 2
    g = np.random.default_rng(77)
    prompts = [g.integers(0, V, n) for n in (40, 60)]

    def fresh():
        m.seq_reset([0, 1])
        pt = torch.zeros(B, 60, dtype=torch.int32)
        for b, pr in enumerate(prompts):
            pt[b, :len(pr)] = torch.as_tensor(pr)
        m.prefill([0, 1], pt.cuda(), [len(pr) for pr in prompts])

    fresh()
    tok = torch.from_numpy(np.concatenate([np.array([[pr[-1]] for pr in prompts]),
                                           g.integers(0, V, (B, N - 1))], 1)).int().cuda()
    lg = m.score([0, 1], tok, parent=TREE).cpu()
    am = lg.argmax(-1)
    for c in (1, 3, 7):                                  # plant a matching branch
        tok[:, c] = am[:, TREE[c]].int().cuda()
        fresh()
        lg = m.score([0, 1], tok, parent=TREE).cpu()
        am = lg.argmax(-1)
    fresh()
    a1, c1, b1 = m.verify_tree_step([0, 1], tok, TREE)
    fresh()
    u = torch.from_numpy(g.random((B, N)).astype(np.float32)).cuda()
    a2, c2, b2 = m.verify_tree_sampled([0, 1], tok, TREE, u, q=None, temperature=1.0, top_k=[1, 1])
    m.sync_status()
    assert torch.equal(a1, a2) and torch.equal(b1, b2) and torch.equal(c1, c2)
    assert int(a1.max()) >= 1
