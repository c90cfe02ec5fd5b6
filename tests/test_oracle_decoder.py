"""Pins of the oracle decoder: hand-computed component values, special cases that
reduce to closed forms, and invariants a plausible mistake would break.
(The pages print no activations, so no pin here comes from them.)"""
import math

import numpy as np
import pytest
import torch

from oracle import decoder as D
from oracle.decoder import CapacityError
from speculative_decoding_verify_step_gb300 import synth
from tests._harness import greedy_decode, greedy_speculative, oracle_model, small_dims


# ---------------------------------------------------------------- components
def test_rmsnorm_hand_value():
    y = D.rmsnorm(np.array([3.0, 4.0]), np.array([1.0, 2.0]), 0.0)
    # mean square 12.5, rms = 3.5355...
    np.testing.assert_allclose(y, [3 / math.sqrt(12.5), 8 / math.sqrt(12.5)], rtol=1e-15)
    y = D.rmsnorm(np.array([1.0, 1.0]), np.array([1.0, 1.0]), 1.0)   # eps inside the root
    np.testing.assert_allclose(y, [1 / math.sqrt(2.0)] * 2, rtol=1e-15)


def test_silu_hand_value():
    np.testing.assert_allclose(D.silu(np.array([0.0, 1.0, -2.0])),
                               [0.0, 0.7310585786300049, -2 / (1 + math.e ** 2)], rtol=1e-14)


def test_rope_hand_values():
    # hd = 4, theta = 10000: inverse frequencies (1, 0.01); pairs (0,2) and (1,3)
    x = np.array([[1.0, 0.0, 0.0, 0.0]])
    np.testing.assert_allclose(D.rope(x, np.array(1), 10000.0)[0],
                               [math.cos(1), 0, math.sin(1), 0], atol=1e-15)
    x = np.array([[0.0, 1.0, 0.0, 0.0]])
    np.testing.assert_allclose(D.rope(x, np.array(3), 10000.0)[0],
                               [0, math.cos(0.03), 0, math.sin(0.03)], atol=1e-15)
    x = np.array([[0.0, 0.0, 1.0, 0.0]])
    np.testing.assert_allclose(D.rope(x, np.array(2), 10000.0)[0],
                               [-math.sin(2), 0, math.cos(2), 0], atol=1e-15)
    rng = np.random.default_rng(0)
    x = rng.normal(size=(3, 8))
    np.testing.assert_allclose(D.rope(x, np.array(0), 500000.0), x, atol=0)


def test_rope_relative_position_property():
    rng = np.random.default_rng(1)
    q, k = rng.normal(size=(1, 128)), rng.normal(size=(1, 128))
    for m, n, s in [(5, 2, 7), (100, 1, 1000), (3, 3, 17)]:
        a = float(D.rope(q, np.array(m), 500000.0)[0] @ D.rope(k, np.array(n), 500000.0)[0])
        b = float(D.rope(q, np.array(m + s), 500000.0)[0] @ D.rope(k, np.array(n + s), 500000.0)[0])
        assert a == pytest.approx(b, rel=1e-10, abs=1e-10)
        assert np.linalg.norm(D.rope(q, np.array(m), 500000.0)) == pytest.approx(np.linalg.norm(q))


def test_attention_hand_values():
    # one query, two keys; scores 0 and 2 ln 3 / sqrt(4) = ln 3 -> weights 1/4, 3/4
    q = np.array([[[1.0, 0, 0, 0]]])
    K = np.array([[[0.0, 0, 0, 0]], [[2 * math.log(3), 0, 0, 0]]])
    V = np.array([[[4.0, 0, 0, 0]], [[0.0, 8, 0, 0]]])
    o = D.attention(q, K, V, np.ones((1, 2), bool))
    np.testing.assert_allclose(o[0, 0], [1.0, 6.0, 0, 0], rtol=1e-14)
    o = D.attention(q, K, V, np.array([[True, False]]))     # the masked key has no weight
    np.testing.assert_allclose(o[0, 0], [4.0, 0, 0, 0], rtol=1e-14)


def test_attention_gqa_mapping():
    # 4 query heads over 2 kv heads: heads 0,1 read kv 0 and heads 2,3 read kv 1
    rng = np.random.default_rng(3)
    q = rng.normal(size=(2, 4, 8))
    K = rng.normal(size=(5, 2, 8))
    V = rng.normal(size=(5, 2, 8))
    vis = np.ones((2, 5), bool)
    o = D.attention(q, K, V, vis)
    o_mha = D.attention(q, np.repeat(K, 2, axis=1), np.repeat(V, 2, axis=1), vis)
    np.testing.assert_allclose(o, o_mha, rtol=1e-14)
    o_wrong = D.attention(q, np.tile(K, (1, 2, 1)), np.tile(V, (1, 2, 1)), vis)
    assert np.abs(o - o_wrong).max() > 1e-3


# ------------------------------------------------------- whole-model special cases
def _zero(weights, names):
    w = dict(weights)
    for n in names:
        w[n] = torch.zeros_like(w[n])
    return w


def test_no_block_output_reduces_to_norm_and_lm_head():
    """With wo = w_down = 0 the residual stream stays the embedding, so the logits
    are rmsnorm(E[t]) g_final W_lm^T for every row."""
    dims = small_dims()
    w = synth.make_weights(dims, 5, gain_jitter=0.1)
    w = _zero(w, [f"layers.{i}.{n}" for i in range(dims.n_layers) for n in ("wo", "w_down")])
    m = oracle_model(dims, weights=w)
    toks = np.array([[3, 7, 11, 2]])
    logits = m.forward([0], toks)
    E = D.bf16_bits_to_f64(m._w["embed"])
    Wl = D.bf16_bits_to_f64(m._w["lm_head"])
    g = w["final_norm"].double().numpy()
    for j, t in enumerate(toks[0]):
        e = E[t]
        ref = (e / math.sqrt(float(np.mean(e * e)) + dims.rms_eps) * g) @ Wl.T
        np.testing.assert_allclose(logits[0, j], ref, rtol=1e-12, atol=1e-14)


def test_single_key_attention_returns_its_value():
    """First token of a sequence: it sees one key (itself), so the attention output is
    its own v; the block output is then h + v Wo^T + ffn."""
    dims = small_dims(n_layers=1, n_kv_heads=4)
    w = synth.make_weights(dims, 6, gain_jitter=0.1)
    w = _zero(w, ["layers.0.w_down"])
    m = oracle_model(dims, weights=w)
    logits, hid = m.forward([0], np.array([[9]]), return_hidden=True)
    f64 = lambda n: D.bf16_bits_to_f64(m._w[n])
    h0 = f64("embed")[9]
    a = D.rmsnorm(h0, w["layers.0.attn_norm"].double().numpy(), dims.rms_eps)
    v = a @ f64("layers.0.wv").T
    h1 = h0 + v @ f64("layers.0.wo").T
    ref = D.rmsnorm(h1, w["final_norm"].double().numpy(), dims.rms_eps)
    np.testing.assert_allclose(hid[0, 0], ref, rtol=1e-11, atol=1e-13)


def test_attention_free_block_is_swiglu_ffn():
    """With wo = 0 a block is h + W_down(silu(W_gate f) * W_up f), f = rmsnorm(h) g_ffn
    (SwiGLU: the gate goes through silu, the up projection does not)."""
    dims = small_dims(n_layers=1)
    w = synth.make_weights(dims, 8, gain_jitter=0.1)
    w = _zero(w, ["layers.0.wo"])
    m = oracle_model(dims, weights=w)
    _, hid = m.forward([0], np.array([[3, 4]]), return_hidden=True)
    f64 = lambda n: D.bf16_bits_to_f64(m._w[n])
    for j, t in enumerate([3, 4]):
        h0 = f64("embed")[t]
        f = D.rmsnorm(h0, w["layers.0.ffn_norm"].double().numpy(), dims.rms_eps)
        g = f @ f64("layers.0.w_gate").T
        u = f @ f64("layers.0.w_up").T
        h1 = h0 + ((g / (1 + np.exp(-g))) * u) @ f64("layers.0.w_down").T
        ref = D.rmsnorm(h1, w["final_norm"].double().numpy(), dims.rms_eps)
        np.testing.assert_allclose(hid[0, j], ref, rtol=1e-11, atol=1e-13)


def test_zero_query_gives_uniform_average_over_visible_keys():
    """wq = 0 makes every score 0: row j of the window averages the v of the L cached
    tokens and of rows 0..j (causal), which pins the mask's extent."""
    dims = small_dims(n_layers=1)
    w = synth.make_weights(dims, 7)
    w = _zero(w, ["layers.0.wq", "layers.0.w_down"])
    m = oracle_model(dims, weights=w)
    prompt = np.array([4, 8, 15, 16, 23, 42, 1])           # 6 cached + pending
    m.prefill([0], [prompt])
    win = np.array([[42 - 41, 5, 6]])
    _, hid = m.forward([0], win, return_hidden=True)
    f64 = lambda n: D.bf16_bits_to_f64(m._w[n])
    allt = np.concatenate([prompt[:-1], win[0]])
    H = f64("embed")[allt]
    A_ = D.rmsnorm(H, w["layers.0.attn_norm"].double().numpy(), dims.rms_eps)
    Vv = (A_ @ f64("layers.0.wv").T).reshape(len(allt), dims.n_kv_heads, dims.head_dim)
    grp = dims.n_heads // dims.n_kv_heads
    for j in range(3):
        mean_v = Vv[:6 + j + 1].mean(axis=0)                 # [Hk, hd]
        o = np.repeat(mean_v, grp, axis=0).reshape(-1)
        h1 = H[6 + j] + o @ f64("layers.0.wo").T
        ref = D.rmsnorm(h1, w["final_norm"].double().numpy(), dims.rms_eps)
        np.testing.assert_allclose(hid[0, j], ref, rtol=1e-11, atol=1e-13)


# ------------------------------------------------------------------ invariants
def test_causality():
    m = oracle_model(small_dims())
    base = np.array([[1, 2, 3, 4, 5]])
    l1 = m.forward([0], base)
    other = base.copy()
    other[0, 3:] = [40, 41]
    l2 = m.forward([0], other)
    np.testing.assert_allclose(l1[0, :3], l2[0, :3], rtol=0, atol=0)
    assert np.abs(l1[0, 3:] - l2[0, 3:]).max() > 1e-6


def test_window_equals_sequential_decode():
    """One forward over W rows == W width-1 forwards with full commits (section 6.1)."""
    dims = small_dims()
    m = oracle_model(dims, gain_jitter=0.1)
    m.prefill([0], [np.array([5, 9, 2, 7, 30, 31, 12])])
    win = np.array([[12, 3, 44, 8, 19]])
    L0 = m.lengths([0])[0]
    lw = m.forward([0], win)
    seq = []
    for j in range(win.shape[1]):
        seq.append(m.forward([0], win[:, j:j + 1])[0, 0])
        m.commit([0], [0], 1)
    np.testing.assert_allclose(lw[0], np.array(seq), rtol=1e-10, atol=1e-12)
    assert m.lengths([0])[0] == L0 + win.shape[1]


def test_batching_equals_each_alone():
    """Selective batching (section 4.2): flattening B sequences changes nothing."""
    dims = small_dims()
    m = oracle_model(dims)
    prompts = [np.arange(1, 70) % 50, np.array([3, 1, 4, 1, 5])]
    m.prefill([0, 1], prompts)
    toks = np.array([[1, 2, 3], [4, 5, 6]])
    both = m.forward([0, 1], toks)
    a = oracle_model(dims)
    a.prefill([0], prompts[:1])
    b = oracle_model(dims)
    b.prefill([1], prompts[1:])
    np.testing.assert_allclose(both[0], a.forward([0], toks[:1])[0], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(both[1], b.forward([1], toks[1:])[0], rtol=1e-11, atol=1e-13)


def test_tree_rows_equal_chain_over_root_path():
    """Each tree node's logits equal the chain forward over its root-to-node path."""
    dims = small_dims()
    m = oracle_model(dims)
    m.prefill([0], [np.array([7, 3, 11, 20])])
    parent = np.array([-1, 0, 0, 1, 1, 2, 2])
    tok = np.array([[20, 5, 6, 7, 8, 9, 10]])
    lt = m.forward([0], tok, parent=parent)
    for node in range(len(parent)):
        path, v = [], node
        while v >= 0:
            path.append(v)
            v = parent[v]
        path = path[::-1]
        lc = m.forward([0], tok[:, path])
        np.testing.assert_allclose(lt[0, node], lc[0, -1], rtol=1e-10, atol=1e-12)
    chain = np.arange(-1, 6)
    np.testing.assert_allclose(m.forward([0], tok[:, :7], parent=chain), m.forward([0], tok[:, :7]),
                               rtol=0, atol=0)


def test_greedy_speculation_equals_greedy_decode():
    """Section 7.4: greedy speculative output is token-for-token the target's greedy
    output, whatever the drafts (random, perfect, or a mix)."""
    dims = small_dims()
    m = oracle_model(dims, gain_jitter=0.1, max_seq_len=256)
    prompts = [np.array([1, 2, 3, 4, 5, 6]), np.array([9, 8, 7])]
    ref = greedy_decode(m, [0, 1], prompts, 24)
    rng = np.random.default_rng(0)
    ref_hist = [list(p) + r for p, r in zip(prompts, ref)]

    def random_draft(h, g):
        return rng.integers(0, dims.vocab, g)

    def perfect_draft(h, g):
        for rh in ref_hist:
            if rh[:len(h)] == h:
                return rh[len(h):len(h) + g] + [0] * max(0, len(h) + g - len(rh))
        raise AssertionError

    def mixed_draft(h, g):
        d = list(perfect_draft(h, g))
        if rng.random() < 0.5:
            d[int(rng.integers(0, g))] = int(rng.integers(0, dims.vocab))
        return d

    for drafter, gamma in [(random_draft, 3), (perfect_draft, 3), (mixed_draft, 4), (perfect_draft, 7)]:
        out, rounds = greedy_speculative(m, [0, 1], prompts, 24, gamma, drafter)
        assert out == ref
        if drafter is perfect_draft:
            assert rounds == -(-24 // (gamma + 1))


def test_kv_after_speculation_equals_plain_decode():
    """Pending-token invariant: after speculative rounds the cache below L equals
    the cache a plain decode of the same committed tokens builds."""
    dims = small_dims()
    prompts = [np.array([5, 4, 3, 2, 1])]
    a = oracle_model(dims)
    rng = np.random.default_rng(1)
    out, _ = greedy_speculative(a, [0], prompts, 20, 3, lambda h, g: rng.integers(0, dims.vocab, g))
    b = oracle_model(dims)
    ref = greedy_decode(b, [0], prompts, 20)
    assert out == ref
    La, Lb = a.lengths([0])[0], b.lengths([0])[0]
    L = min(La, Lb)
    for t in range(L):
        pa, oa = a.kv.slot(0, t)
        pb, ob = b.kv.slot(0, t)
        np.testing.assert_allclose(a.kv.k[:, pa, :, oa], b.kv.k[:, pb, :, ob], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(a.kv.v[:, pa, :, oa], b.kv.v[:, pb, :, ob], rtol=1e-10, atol=1e-12)


# ------------------------------------------------------------ pages and commit
def test_page_tables_scripted():
    dims = small_dims(n_layers=1)
    m = oracle_model(dims, max_batch=3, max_seq_len=256, num_pages=8)
    m.prefill([0], [np.zeros(65, np.int64)])          # L = 64: one full page
    assert m.kv.table[0] == [0] and m.lengths([0])[0] == 64
    m.prefill([1], [np.zeros(10, np.int64)])          # L = 9
    assert m.kv.table[1] == [1]
    m.forward([0, 1], np.zeros((2, 4), np.int64))     # seq 0 needs slots 64..67: page 2
    assert m.kv.table[0] == [0, 2] and m.kv.table[1] == [1]
    m.commit([0, 1], [0, 3], 4)                       # seq 0: L = 65; seq 1: L = 13
    assert m.kv.table[0] == [0, 2] and m.lengths([0, 1]).tolist() == [65, 13]
    m.forward([0], np.zeros((1, 4), np.int64))
    m.commit([0], [0], 4)
    assert m.kv.table[0] == [0, 2]
    m.reset([0])
    assert m.kv.free[:3] == [True, False, True]
    m.prefill([2], [np.zeros(130, np.int64)])         # L = 129: pages 0, 2, 3
    assert m.kv.table[2] == [0, 2, 3]


def test_commit_frees_pages_beyond_length():
    dims = small_dims(n_layers=1)
    m = oracle_model(dims, max_batch=1, max_seq_len=256, num_pages=4)
    m.prefill([0], [np.zeros(62, np.int64)])          # L = 61
    m.forward([0], np.zeros((1, 8), np.int64))        # slots 61..68 -> pages 0, 1
    assert m.kv.table[0] == [0, 1]
    m.commit([0], [1], 8)                             # L = 63: page 1 holds nothing kept
    assert m.kv.table[0] == [0] and m.kv.free[1]
    m.forward([0], np.zeros((1, 2), np.int64))
    m.commit([0], [1], 2)                             # L = 65: keeps page 1
    assert m.kv.table[0] == [0, 1]
    # a commit landing exactly on a page boundary frees the page that starts there
    m2 = oracle_model(dims, max_batch=1, max_seq_len=256, num_pages=4)
    m2.prefill([0], [np.zeros(62, np.int64)])         # L = 61
    m2.forward([0], np.zeros((1, 8), np.int64))
    m2.commit([0], [2], 8)                            # L = 64: page 1 starts at slot 64
    assert m2.kv.table[0] == [0] and m2.lengths([0])[0] == 64


def test_capacity_errors():
    dims = small_dims(n_layers=1)
    m = oracle_model(dims, max_batch=2, max_seq_len=128, num_pages=2)
    m.prefill([0], [np.zeros(100, np.int64)])
    with pytest.raises(CapacityError):
        m.prefill([1], [np.zeros(10, np.int64)])     # pool exhausted
    m2 = oracle_model(dims, max_batch=1, max_seq_len=64, num_pages=4)
    m2.prefill([0], [np.zeros(60, np.int64)])
    with pytest.raises(CapacityError):
        m2.forward([0], np.zeros((1, 8), np.int64))  # beyond max_seq_len


def test_tree_commit_compacts_path():
    """After a tree round the accepted path's KV sits at L+1..L+n and equals the KV a
    chain round over the same tokens writes."""
    dims = small_dims()
    m = oracle_model(dims)
    m.prefill([0], [np.array([7, 3, 11, 20])])
    L = m.lengths([0])[0]
    parent = np.array([-1, 0, 0, 1, 1, 2, 2])
    tok = np.array([[20, 5, 6, 7, 8, 9, 10]])
    m.forward([0], tok, parent=parent)
    path = np.array([[2, 6]])
    m.commit_tree([0], path)
    assert m.lengths([0])[0] == L + 3
    c = oracle_model(dims)
    c.prefill([0], [np.array([7, 3, 11, 20])])
    c.forward([0], np.array([[20, 6, 10]]))
    c.commit([0], [2], 3)
    for t in range(L + 3):
        pa, oa = m.kv.slot(0, t)
        pc, oc = c.kv.slot(0, t)
        np.testing.assert_allclose(m.kv.k[:, pa, :, oa], c.kv.k[:, pc, :, oc], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(m.kv.v[:, pa, :, oa], c.kv.v[:, pc, :, oc], rtol=1e-10, atol=1e-12)
