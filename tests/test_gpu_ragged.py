"""Ragged verify on the GPU vs the oracle: per-sequence verify lengths in one batch
(the accounting page's example, section 四: lengths 6, 2, 1, 4 with gamma + 1 = 6),
cap-accept (fixed-width forward, capped acceptance) and compact (packed rows)."""
import numpy as np
import pytest
import torch

from oracle import accept as A
from speculative_decoding_verify_step_gb300 import synth
from tests._gpu import cuda_model, need_gpu, oracle_for, stochastic_margin, top2_gap

pytestmark = pytest.mark.gpu
LENS = [6, 2, 1, 4]
KW = dict(max_batch=4, max_width=16, max_seq_len=512, num_pages=40)


@pytest.fixture(scope="module")
def tiny():
    need_gpu()
    w = synth.make_weights(synth.TINY, seed=1, gain_jitter=0.1)
    m = cuda_model(synth.TINY, w, **KW)
    yield w, m
    m.close()


def _setup(w, m, seed):
    g = np.random.default_rng(seed)
    prompts = [g.integers(0, synth.TINY.vocab, n) for n in (70, 40, 65, 50)]
    ids = list(range(4))
    m.seq_reset(ids)
    tok = torch.zeros(4, 70, dtype=torch.int32)
    for b, p in enumerate(prompts):
        tok[b, :len(p)] = torch.as_tensor(p)
    m.prefill(ids, tok.cuda(), [len(p) for p in prompts])
    o = oracle_for(synth.TINY, w, **KW)
    o.prefill(ids, prompts)
    return ids, prompts, o


@pytest.mark.parametrize("mode", ["cap", "compact"])
@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_ragged_rounds(tiny, mode, temp):
    compared = sum(_ragged_round(tiny, mode, temp, seed) for seed in (21, 22, 23))
    assert compared >= 4


def _ragged_round(tiny, mode, temp, seed):
    """One ragged round; returns how many sequences were clear of the margins (and
    therefore compared bit for bit)."""
    from speculative_decoding_verify_step_gb300 import spec
    w, m = tiny
    ids, prompts, o = _setup(w, m, seed=seed + int(temp))
    gamma, V = 5, synth.TINY.vocab
    g = np.random.default_rng(seed)
    tok = np.concatenate([np.array([[p[-1]] for p in prompts]), g.integers(0, V, (4, gamma))], axis=1)
    # make most drafts the target's greedy choice so acceptance is non-trivial (a
    # second oracle drafts, so the scoring oracle's pages follow the rounds only)
    _, _, od = _setup(w, m, seed=seed + int(temp))
    ref_full = od.forward(ids, tok)
    for b in range(4):
        for i in range(1, gamma + 1):
            if g.random() < 0.7:
                tok[b, i] = ref_full[b, i - 1].argmax()
                ref_full = od.forward(ids, tok)
    q = synth.dirichlet1((4, gamma, V), seed=5).numpy().astype(np.float32)
    for b in range(4):                       # drafts then carry most of q's mass
        for i in range(gamma):
            q[b, i] = 0.5 * q[b, i]
            q[b, i, tok[b, i + 1]] += 0.5
    u = synth.uniforms((4, gamma + 1), seed=6).numpy()
    # oracle: each sequence scores its own window (cap: the full width; compact: its length)
    n_ref, com_ref = np.zeros(4, np.int64), np.full((4, gamma + 1), -1, np.int64)
    clear = np.ones(4, bool)
    for b, s in enumerate(ids):
        Lb = LENS[b]
        width = gamma + 1 if mode == "cap" else Lb
        logits = o.forward([s], tok[b:b + 1, :width])[:, :Lb]
        if temp == 0.0:
            n, com, _ = A.accept_greedy(logits, tok[b:b + 1, 1:Lb])
            clear[b] = (top2_gap(logits)[0, :n[0] + 1] > 1e-2).all()
        else:
            p = A.target_probs(logits, temp)
            n, com, _, _ = A.accept_stochastic(p, q[b:b + 1, :Lb - 1], tok[b:b + 1, 1:Lb], u[b:b + 1, :Lb])
            clear[b] = stochastic_margin(p, q[b:b + 1, :Lb - 1], tok[b:b + 1, 1:Lb], u[b:b + 1, :Lb], n)[0]
        n_ref[b] = n[0]
        com_ref[b, :Lb] = com[0]
    lens = torch.tensor(LENS, dtype=torch.int32).cuda()
    if mode == "cap":
        t_in = torch.from_numpy(tok).cuda()
        md = spec.RAGGED_CAP_ACCEPT
    else:
        t_in = torch.from_numpy(np.concatenate([tok[b, :LENS[b]] for b in range(4)])).cuda()
        md = spec.RAGGED_COMPACT
    kw = {} if temp == 0.0 else dict(q=torch.from_numpy(q).cuda(), u=torch.from_numpy(u).cuda())
    acc, com, bon = m.verify_ragged(ids, t_in, lens, md, temperature=temp, gamma=gamma, **kw)
    m.sync_status()
    acc, com = acc.cpu().numpy(), com.cpu().numpy()
    for b in range(4):
        assert acc[b] <= LENS[b] - 1
        if clear[b]:
            assert acc[b] == n_ref[b], (b, acc[b], n_ref[b])
            np.testing.assert_array_equal(com[b], com_ref[b])
    if clear.all():
        o.commit(ids, n_ref, gamma + 1)
        lens_m, pt = m.kv_state(ids)
        assert lens_m == o.lengths(ids).tolist()
        np.testing.assert_array_equal(np.array(pt), o.kv.page_table_array(ids))
    return int(clear.sum())


def test_cap_accept_at_full_length_equals_verify(tiny):
    """verify_lens = gamma + 1 everywhere: cap-accept is the static verify round."""
    from speculative_decoding_verify_step_gb300 import spec
    w, m = tiny
    ids, prompts, _ = _setup(w, m, seed=30)
    gamma = 3
    g = np.random.default_rng(4)
    tok = torch.from_numpy(np.concatenate([np.array([[p[-1]] for p in prompts]),
                                           g.integers(0, synth.TINY.vocab, (4, gamma))], axis=1)).int().cuda()
    a1, c1, b1 = m.verify_ragged(ids, tok, [gamma + 1] * 4, spec.RAGGED_CAP_ACCEPT)
    ids2, _, _ = _setup(w, m, seed=30)
    a2, c2, b2 = m.verify_step(ids2, tok)
    assert torch.equal(a1, a2) and torch.equal(c1, c2) and torch.equal(b1, b2)


def test_compact_length_mismatch_is_reported(tiny):
    from speculative_decoding_verify_step_gb300 import spec
    w, m = tiny
    ids, prompts, _ = _setup(w, m, seed=31)
    tok = torch.zeros(13, dtype=torch.int32).cuda()         # sum(LENS) = 13
    bad = torch.tensor([6, 2, 2, 4], dtype=torch.int32).cuda()  # sums to 14
    m.verify_ragged(ids, tok, bad, spec.RAGGED_COMPACT, gamma=5)
    with pytest.raises(spec.SpecError) as e:
        m.sync_status()
    assert e.value.status == 1
