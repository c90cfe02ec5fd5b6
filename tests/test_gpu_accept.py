"""Standalone acceptance on the GPU vs the oracle: bit-exact on identical p, q, u."""
import numpy as np
import pytest
import torch

from oracle import accept as A
from speculative_decoding_verify_step_gb300 import synth
from tests._gpu import need_gpu

pytestmark = pytest.mark.gpu


def _case(B, gamma, V, seed, lam=0.5, zero_q=False, eq=False, peaked=False):
    rng = np.random.default_rng(seed)
    W = gamma + 1
    logits = rng.normal(size=(B, W, V)) * (4.0 if peaked else 1.3)
    p = A.target_probs(logits, 1.0)
    D = synth.dirichlet1((B, max(gamma, 1), V), seed=seed + 1).numpy()
    q = ((1 - lam) * p[:, :gamma].astype(np.float64) + lam * D[:, :gamma]).astype(np.float32)
    if eq:
        q = p[:, :gamma].copy()
    if zero_q and gamma > 0:
        q[:, :, ::7] = 0.0
    x = np.zeros((B, gamma), np.int64)
    for b in range(B):
        for i in range(gamma):
            c = np.cumsum(q[b, i].astype(np.float64))
            x[b, i] = min(int(np.searchsorted(c, rng.random() * c[-1], side="right")), V - 1)
    u = synth.uniforms((B, W), seed=seed + 2).numpy()
    u[0, :] = 0.0
    if B > 1:
        u[1, :] = np.float32(1 - 2 ** -24)
    return p, q, x, u


@pytest.mark.parametrize("B,gamma,V,kw", [
    (64, 3, 1024, {}),
    (64, 7, 1024, {"lam": 0.2}),
    (32, 4, 128256, {"lam": 0.8}),
    (16, 0, 128256, {}),
    (48, 3, 1024, {"zero_q": True}),
    (32, 5, 1000, {"eq": True}),
    (32, 15, 4096, {"peaked": True}),
    (1, 1, 3, {}),
])
def test_accept_probs_bitexact(B, gamma, V, kw):
    need_gpu()
    from speculative_decoding_verify_step_gb300 import spec
    p, q, x, u = _case(B, gamma, V, seed=B * 100 + gamma, **kw)
    n_ref, com_ref, tok_ref, _ = A.accept_stochastic(p, q, x, u)
    dev = torch.device("cuda")
    acc, com, bon = spec.spec_accept_probs(torch.from_numpy(p).to(dev),
                                           torch.from_numpy(q).to(dev) if gamma else None,
                                           torch.from_numpy(x).to(dev) if gamma else None,
                                           torch.from_numpy(u).to(dev))
    np.testing.assert_array_equal(acc.cpu().numpy(), n_ref)
    np.testing.assert_array_equal(com.cpu().numpy(), com_ref)
    np.testing.assert_array_equal(bon.cpu().numpy(), tok_ref)


def test_accept_probs_massless_rows_give_token_0():
    """Rows of p without mass on the 2^-40 grid (all zeros, or every entry below
    2^-40) are not distributions; the draw gives token 0, as the oracle does, both
    after a rejection and as the bonus.  V = 128256 spans the 8-CTA cluster."""
    need_gpu()
    from speculative_decoding_verify_step_gb300 import spec
    for V in (1024, 128256):
        p, q, x, u = _case(6, 3, V, seed=77)
        p[0] = 0.0                                   # every row: rejected (p(x) = 0), then no mass
        p[1, 3] = 0.0                                # the bonus row only
        p[2] = np.float32(2.0 ** -42)                # mass below the grid everywhere
        p[3, 1:] = 0.0
        u[1, :3] = 0.0                               # sequence 1 accepts its drafts where p(x) > 0
        n_ref, com_ref, tok_ref, _ = A.accept_stochastic(p, q, x, u)
        d = lambda a: torch.from_numpy(a).cuda()
        acc, com, bon = spec.spec_accept_probs(d(p), d(q), d(x), d(u))
        np.testing.assert_array_equal(acc.cpu().numpy(), n_ref)
        np.testing.assert_array_equal(com.cpu().numpy(), com_ref)
        np.testing.assert_array_equal(bon.cpu().numpy(), tok_ref)
        assert tok_ref[0] == 0 and tok_ref[2] == 0


def test_accept_probs_exercise3_law():
    """Exercise 3 through the GPU rule: over a grid of uniforms the output frequencies
    equal p = (0.5, 0.3, 0.2) to the grid resolution."""
    need_gpu()
    from speculative_decoding_verify_step_gb300 import spec
    n = 1 << 16
    p = np.tile(np.array([[0.5, 0.3, 0.2], [0.5, 0.3, 0.2]], np.float32), (n, 1, 1))
    q = np.tile(np.array([[0.2, 0.6, 0.2]], np.float32), (n, 1, 1))
    rng = np.random.default_rng(0)
    x = (np.cumsum([0.2, 0.6, 0.2])[None] < rng.random((n, 1))).sum(-1)[:, None]
    u = rng.random((n, 2)).astype(np.float32)
    dev = torch.device("cuda")
    acc, com, _ = spec.spec_accept_probs(*(torch.from_numpy(a).to(dev) for a in (p, q, x, u)))
    first = com[:, 0].cpu().numpy()
    freq = np.bincount(first, minlength=3) / n
    np.testing.assert_allclose(freq, [0.5, 0.3, 0.2], atol=4 * np.sqrt(0.25 / n))
    assert acc.float().mean().item() == pytest.approx(0.7, abs=4 * np.sqrt(0.21 / n))


@pytest.mark.parametrize("B,gamma,V", [(64, 3, 1024), (16, 7, 128256), (8, 0, 1024)])
def test_accept_greedy_bitexact(B, gamma, V):
    need_gpu()
    from speculative_decoding_verify_step_gb300 import spec
    rng = np.random.default_rng(B + gamma)
    W = gamma + 1
    logits = rng.normal(size=(B, W, V)).astype(np.float32)
    logits[:, :, 5] = logits.max(-1) + 1.0          # rows with a tie at the top: index 5 vs 9
    logits[::2, :, 9] = logits[::2, :, 5]
    am = logits.argmax(-1)
    x = np.where(rng.random((B, gamma)) < 0.6, am[:, :gamma], rng.integers(0, V, (B, gamma)))
    n_ref, com_ref, bon_ref = A.accept_greedy(logits, x)
    dev = torch.device("cuda")
    acc, com, bon = spec.spec_accept_greedy(torch.from_numpy(logits).to(dev),
                                            torch.from_numpy(x).to(dev) if gamma else None)
    np.testing.assert_array_equal(acc.cpu().numpy(), n_ref)
    np.testing.assert_array_equal(com.cpu().numpy(), com_ref)
    np.testing.assert_array_equal(bon.cpu().numpy(), bon_ref)
