"""GPU-test helpers: CUDA models built from the same seeded weights as the oracle."""
import numpy as np
import pytest
import torch

from oracle import accept as A
from oracle.decoder import OracleDecoder, weights_to_numpy


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")


def cuda_model(dims, weights, **kw):
    from speculative_decoding_verify_step_gb300 import spec
    m = spec.SpecModel(dims, **kw)
    m.load_weights((k, v.cuda()) for k, v in weights.items())
    return m


def oracle_for(dims, weights, **kw):
    kw = {k: v for k, v in kw.items() if k in ("max_batch", "max_seq_len", "num_pages")}
    return OracleDecoder(dims, weights_to_numpy(weights), **kw)


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.abs(got - ref).max() / np.abs(ref).max())


def top2_gap(logits):
    t = np.sort(np.asarray(logits, np.float64), axis=-1)
    return t[..., -1] - t[..., -2]


def greedy_clear(ref_logits, n_ref, margin=1e-2):
    """A greedy round's decisions are fixed by the reference logits when every row the
    decision reads (rows 0..n) has a top-2 gap above the margin."""
    gap = top2_gap(ref_logits)
    B = gap.shape[0]
    return np.array([(gap[b, :n_ref[b] + 1] > margin).all() for b in range(B)])


def stochastic_margin(p, q, x, u, n, margin=1e-2, draw_margin=1e-4):
    """Clear when every accept test the round took has |u - p/q| > margin and the final
    draw's threshold t sits more than margin x (its step's width) and more than
    draw_margin x S from each edge of its CDF step."""
    B, W, V = p.shape
    clear = np.ones(B, bool)
    for b in range(B):
        for i in range(1, min(int(n[b]) + 1, W - 1) + 1):
            xi = int(x[b, i - 1])
            qx, px = float(q[b, i - 1, xi]), float(p[b, i - 1, xi])
            ratio = px / qx if qx > 0 else np.inf
            if abs(float(u[b, i - 1]) - ratio) <= margin:
                clear[b] = False
        row = int(n[b])
        r = A.residual(p[b, row], q[b, row]) if row < W - 1 else p[b, row]
        R = A.fixed_point_mass(r).astype(np.float64)
        S = R.sum()
        if S == 0:
            clear[b] = False
            continue
        # the chosen step [C_{v-1}, C_v) of the integer CDF: t must sit more than
        # margin x (step width) inside it, and more than draw_margin x S from either
        # edge (the CDF drift that logit differences can cause: 1e-4 S for logits of
        # std ~0.3, up to ~1e-2 S for logits of std ~5)
        t = np.floor(float(u[b, W - 1]) * 2 ** 24) * S / 2 ** 24
        edges = np.cumsum(R)
        v = int(np.searchsorted(edges, t, side="right"))
        lo = edges[v - 1] if v > 0 else 0.0
        hi = edges[v]
        gapd = min(t - lo, hi - t)
        if gapd <= margin * (hi - lo) or gapd <= draw_margin * S:
            clear[b] = False
    return clear
