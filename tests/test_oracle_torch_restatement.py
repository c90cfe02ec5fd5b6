"""Pin of the oracle decoder's forward against an independent restatement built from
PyTorch library routines (CPU, float64): torch's RMSNorm, its scaled-dot-product
attention with a boolean mask and grouped kv heads, SiLU, and rotary embedding
written as a complex rotation (torch.polar) instead of the oracle's
cos/sin pair arithmetic.

The restatement scores a whole sequence in one pass (cached prefix and window
together), so it also pins the oracle's paged cache, its prefill windows and the
positions it gives the window rows (chain: L + j; tree: L + depth).  The pages
print no decoder activations; the readings restated here are the standard Llama
form named by the workload: RMSNorm x / sqrt(mean x^2 + eps) * g, half-split
rotary pairs (i, i + hd/2) at absolute positions with inverse frequency
theta^(-2i/hd), scale 1/sqrt(hd), query head h reading kv head h // (Hq/Hkv),
SwiGLU W_down(silu(W_gate f) * W_up f), untied embedding and LM head.

Planted mistakes in where the oracle applies RoPE to the keys (not rotated;
rotated one position late) must fail the comparison."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import decoder as D
from oracle.accept import tree_ancestors, tree_depths
from speculative_decoding_verify_step_gb300 import synth
from tests._harness import oracle_model, small_dims

TOL = 1e-9      # float64 on both sides; only the summation order differs


def _w(weights, name):
    t = weights[name]
    return t.to(torch.float64)


def _rotate(x, pos, theta):
    """x [T, H, hd], pos [T]: pair (x_i, x_{i+hd/2}) as the complex number
    x_i + i x_{i+hd/2}, multiplied by exp(i pos theta^(-2i/hd))."""
    hd = x.shape[-1]
    half = hd // 2
    inv = torch.pow(torch.tensor(float(theta), dtype=torch.float64),
                    -torch.arange(0, hd, 2, dtype=torch.float64) / hd)          # [half]
    ang = pos.to(torch.float64)[:, None] * inv[None, :]                       # [T, half]
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]                  # [T, 1, half]
    z = torch.complex(x[..., :half], x[..., half:]) * rot
    return torch.cat([z.real, z.imag], dim=-1)


def torch_logits(dims, weights, tokens, pos, visible):
    """Logits of every row of one sequence.  tokens [T], pos [T] (rotary positions),
    visible [T, T] bool (row r may attend to key c)."""
    tok = torch.as_tensor(np.asarray(tokens), dtype=torch.long)
    pos = torch.as_tensor(np.asarray(pos), dtype=torch.long)
    mask = torch.as_tensor(np.asarray(visible), dtype=torch.bool)
    T = tok.numel()
    d, Hq, Hk, hd = dims.d_model, dims.n_heads, dims.n_kv_heads, dims.head_dim
    h = _w(weights, "embed")[tok]                                            # [T, d]
    for li in range(dims.n_layers):
        p = f"layers.{li}."
        a = F.rms_norm(h, (d,), _w(weights, p + "attn_norm"), eps=dims.rms_eps)
        q = _rotate((a @ _w(weights, p + "wq").T).view(T, Hq, hd), pos, dims.rope_theta)
        k = _rotate((a @ _w(weights, p + "wk").T).view(T, Hk, hd), pos, dims.rope_theta)
        v = (a @ _w(weights, p + "wv").T).view(T, Hk, hd)
        o = F.scaled_dot_product_attention(q.transpose(0, 1)[None], k.transpose(0, 1)[None],
                                           v.transpose(0, 1)[None], attn_mask=mask, enable_gqa=True)
        h = h + o[0].transpose(0, 1).reshape(T, Hq * hd) @ _w(weights, p + "wo").T
        f = F.rms_norm(h, (d,), _w(weights, p + "ffn_norm"), eps=dims.rms_eps)
        h = h + (F.silu(f @ _w(weights, p + "w_gate").T) * (f @ _w(weights, p + "w_up").T)) @ _w(weights, p + "w_down").T
    return F.rms_norm(h, (d,), _w(weights, "final_norm"), eps=dims.rms_eps) @ _w(weights, "lm_head").T


def sequence_layout(L, parent):
    """Positions and visibility of a cached prefix of L tokens followed by a window
    (parent[0] = -1; a chain is parent[j] = j - 1)."""
    W = len(parent)
    depth = tree_depths(parent)
    anc = tree_ancestors(parent)
    pos = np.concatenate([np.arange(L), L + depth])
    vis = np.zeros((L + W, L + W), bool)
    vis[:L, :L] = np.tril(np.ones((L, L), bool))
    vis[L:, :L] = True
    for j in range(W):
        for i in anc[j]:
            vis[L + j, L + i] = True
    return pos, vis


def oracle_vs_torch(dims, weights, prompt, window, parent):
    """Largest relative difference between the oracle's window logits (after a
    prefill of the prompt) and the restatement's over the same token sequence."""
    m = oracle_model(dims, weights=weights, max_seq_len=512, num_pages=32)
    m.prefill([0], [prompt])
    got = m.forward([0], np.asarray(window)[None], parent=None if parent is None else np.asarray(parent))[0]
    par = np.arange(-1, len(window) - 1) if parent is None else np.asarray(parent)
    L = len(prompt) - 1
    pos, vis = sequence_layout(L, par)
    ref = torch_logits(dims, weights, np.concatenate([prompt[:-1], window]), pos, vis)[L:].numpy()
    return float(np.abs(got - ref).max() / np.abs(ref).max())


TREE7 = [-1, 0, 0, 1, 1, 2, 2]


def _case(dims, seed, L=70):
    w = synth.make_weights(dims, seed, gain_jitter=0.1)
    g = np.random.default_rng(seed)
    prompt = g.integers(0, dims.vocab, L + 1)
    window = np.concatenate([[prompt[-1]], g.integers(0, dims.vocab, 6)])
    return w, prompt, window


@pytest.mark.parametrize("parent", [None, TREE7], ids=["chain", "tree"])
@pytest.mark.parametrize("which", ["gqa", "tiny"])
def test_oracle_forward_equals_torch_restatement(which, parent):
    dims = small_dims(rope_theta=500.0) if which == "gqa" else synth.TINY
    w, prompt, window = _case(dims, 31)
    assert oracle_vs_torch(dims, w, prompt, window, parent) < TOL


def test_positions_matter_in_this_pin():
    """The case above is sensitive to relative positions: moving the window rows
    three positions away from the prefix changes the logits clearly, while moving
    every position by the same amount changes nothing (rotary scores depend on the
    offset between query and key only)."""
    dims = small_dims(rope_theta=500.0)
    w, prompt, window = _case(dims, 31)
    L = len(prompt) - 1
    pos, vis = sequence_layout(L, np.arange(-1, len(window) - 1))
    toks = np.concatenate([prompt[:-1], window])
    a = torch_logits(dims, w, toks, pos, vis)[L:]
    moved = pos.copy()
    moved[L:] += 3
    b = torch_logits(dims, w, toks, moved, vis)[L:]
    assert float((a - b).abs().max() / a.abs().max()) > 1e-3
    c = torch_logits(dims, w, toks, pos + 5, vis)[L:]
    assert float((a - c).abs().max() / a.abs().max()) < TOL


def _planted_rope(kind):
    """The oracle's forward calls rope(q) then rope(k) in every layer; this stand-in
    keeps the query rotation and plants a mistake in the key rotation."""
    calls = {"n": 0}
    right = D.rope

    def rope(x, pos, theta):
        calls["n"] += 1
        if calls["n"] % 2 == 1:
            return right(x, pos, theta)
        if kind == "keys_not_rotated":
            return x.copy()
        return right(x, np.asarray(pos) + 1, theta)       # keys one position late
    return rope


@pytest.mark.parametrize("kind", ["keys_not_rotated", "keys_one_late"])
def test_planted_key_rotation_mistakes_fail(monkeypatch, kind):
    dims = small_dims(rope_theta=500.0)
    w, prompt, window = _case(dims, 31)
    monkeypatch.setattr(D, "rope", _planted_rope(kind))
    assert oracle_vs_torch(dims, w, prompt, window, None) > 1e-4
