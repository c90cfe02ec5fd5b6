"""GPU verify round vs the oracle on the tiny 2-layer decoder (d 256, 4x64 heads,
SwiGLU 1024, vocab 1024): forward parity, KV/page tables, greedy and sampled
rounds, decode steps, the token tree, and error paths."""
import numpy as np
import pytest
import torch

from oracle import accept as A
from speculative_decoding_verify_step_gb300 import synth
from tests._gpu import cuda_model, greedy_clear, need_gpu, oracle_for, rel_err, stochastic_margin

pytestmark = pytest.mark.gpu

TOL = 1e-2          # max-abs error relative to max|ref| (bf16 weights, fp32 accumulation)
KW = dict(max_batch=4, max_width=16, max_seq_len=512, num_pages=40)


@pytest.fixture(scope="module")
def tiny():
    need_gpu()
    w = synth.make_weights(synth.TINY, seed=1, gain_jitter=0.1)
    m = cuda_model(synth.TINY, w, **KW)
    yield w, m
    m.close()


def _fresh(w, m, prompts):
    ids = list(range(len(prompts)))
    m.seq_reset(ids)
    L = max(len(p) for p in prompts)
    tok = torch.zeros(len(prompts), L, dtype=torch.int32)
    for b, p in enumerate(prompts):
        tok[b, :len(p)] = torch.as_tensor(p)
    m.prefill(ids, tok.cuda(), [len(p) for p in prompts])
    o = oracle_for(synth.TINY, w, **KW)
    o.prefill(ids, prompts)
    return ids, o


def _prompts(lens, seed):
    g = np.random.default_rng(seed)
    return [g.integers(0, synth.TINY.vocab, n) for n in lens]


def test_forward_logits_and_kv(tiny):
    w, m = tiny
    prompts = _prompts([64, 37], 2)
    ids, o = _fresh(w, m, prompts)
    lens, pt = m.kv_state(ids)
    assert lens == [63, 36]
    np.testing.assert_array_equal(np.array(pt), o.kv.page_table_array(ids))
    tok = np.stack([np.concatenate([[p[-1]], d]) for p, d in zip(prompts, _prompts([3, 3], 3))])
    got = m.score(ids, torch.from_numpy(tok).cuda()).cpu().numpy()
    ref = o.forward(ids, tok)
    assert rel_err(got, ref) < TOL
    # cached KV (bf16) against the oracle's (fp64), all layers, prompt and window slots
    for layer in range(synth.TINY.n_layers):
        for b, s in enumerate(ids):
            n = len(prompts[b]) - 1 + 4
            k, v = m.read_kv(layer, s, 0, n)
            kr = np.stack([o.kv.k[layer, o.kv.slot(s, t)[0], :, o.kv.slot(s, t)[1]] for t in range(n)])
            vr = np.stack([o.kv.v[layer, o.kv.slot(s, t)[0], :, o.kv.slot(s, t)[1]] for t in range(n)])
            assert rel_err(k.float().numpy(), kr) < TOL
            assert rel_err(v.float().numpy(), vr) < TOL


@pytest.mark.parametrize("W", [1, 2, 5, 8, 16])
def test_window_widths(tiny, W):
    w, m = tiny
    prompts = _prompts([130, 64], 10 + W)      # crosses page boundaries; ragged tail
    ids, o = _fresh(w, m, prompts)
    tok = np.stack([np.concatenate([[p[-1]], d]) for p, d in zip(prompts, _prompts([W - 1] * 2, 4))])
    got = m.score(ids, torch.from_numpy(tok).cuda()).cpu().numpy()
    ref = o.forward(ids, tok)
    assert rel_err(got, ref) < TOL


def test_greedy_rounds_teacher_forced(tiny, margins):
    """32 greedy verify rounds (gamma = 3, B = 2) with mixed drafts.  Where every row the
    decision reads has a top-2 gap > 1e-2 the accepted count and committed tokens are
    identical; near-ties are counted and the GPU state is re-synchronised to the oracle."""
    w, m = tiny
    prompts = _prompts([64, 64], 5)
    ids, o = _fresh(w, m, prompts)
    hist = [list(map(int, p)) for p in prompts]
    rng = np.random.default_rng(6)
    gamma, compared, near = 3, 0, 0
    for r in range(32):
        # drafts: the oracle's own greedy continuation, each draft corrupted w.p. 1/4
        tok = np.zeros((2, gamma + 1), np.int64)
        tok[:, 0] = [h[-1] for h in hist]
        for i in range(1, gamma + 1):
            nxt = o.forward(ids, tok[:, :i])[:, i - 1].argmax(-1)
            bad = rng.random(2) < 0.25
            tok[:, i] = np.where(bad, rng.integers(0, synth.TINY.vocab, 2), nxt)
        ref = o.forward(ids, tok)
        n_ref, com_ref, _ = A.accept_greedy(ref, tok[:, 1:])
        acc, com, bon = m.verify_step(ids, torch.from_numpy(tok).cuda())
        got_logits = m.debug_logits(2 * (gamma + 1)).cpu().numpy().reshape(ref.shape)
        assert rel_err(got_logits, ref) < TOL
        clear = greedy_clear(ref, n_ref)
        acc, com = acc.cpu().numpy(), com.cpu().numpy()
        for b in range(2):
            if clear[b]:
                compared += 1
                assert acc[b] == n_ref[b]
                np.testing.assert_array_equal(com[b], com_ref[b])
            else:
                near += 1
        o.commit(ids, n_ref, gamma + 1)
        for b in range(2):
            hist[b].extend(int(t) for t in com_ref[b, :n_ref[b] + 1])
        if not (clear.all() and (acc == n_ref).all()):
            ids, o2 = _fresh(w, m, [np.array(h) for h in hist])   # re-sync both sides
            o = o2
        else:
            lens, pt = m.kv_state(ids)
            assert lens == o.lengths(ids).tolist()
            np.testing.assert_array_equal(np.array(pt), o.kv.page_table_array(ids))
    margins(compared, near)
    assert compared >= 40, (compared, near)


def _draft_mixture(o, ids, pending, gamma, lam, temp, seed):
    """Drafts x_i ~ q_i = (1-lam) p_i + lam Dir(1), p_i the oracle target at the draft
    prefix (an untimed autoregressive target pass)."""
    B = len(ids)
    V = synth.TINY.vocab
    rng = np.random.default_rng(seed)
    D = synth.dirichlet1((B, gamma, V), seed=seed).numpy()
    tok = np.zeros((B, gamma + 1), np.int64)
    tok[:, 0] = pending
    q = np.zeros((B, gamma, V), np.float32)
    for i in range(gamma):
        logits = o.forward(ids, tok[:, :i + 1])
        p = A.target_probs(logits[:, i], temp).astype(np.float64)
        qi = (1 - lam) * p + lam * D[:, i]
        q[:, i] = qi.astype(np.float32)
        for b in range(B):
            c = np.cumsum(q[b, i].astype(np.float64))
            tok[b, i + 1] = min(int(np.searchsorted(c, rng.random() * c[-1], side="right")), V - 1)
    return tok, q


@pytest.mark.parametrize("lam,temp", [(0.5, 1.0), (0.2, 0.7)])
def test_sampled_rounds(tiny, margins, lam, temp):
    """Sampled verify rounds (gamma = 3): bit-exact accepted counts and committed
    tokens wherever the oracle's decisions are clear of the 1e-2 margins."""
    w, m = tiny
    prompts = _prompts([64, 64], 7)
    ids, o = _fresh(w, m, prompts)
    gamma, compared, near = 3, 0, 0
    pending = np.array([p[-1] for p in prompts])
    hist = [list(map(int, p)) for p in prompts]
    for r in range(16):
        tok, q = _draft_mixture(o, ids, pending, gamma, lam, temp, seed=100 + r)
        u = synth.uniforms((2, gamma + 1), seed=200 + r).numpy()
        logits = o.forward(ids, tok)
        p = A.target_probs(logits, temp)
        n_ref, com_ref, tok_ref, _ = A.accept_stochastic(p, q, tok[:, 1:], u)
        acc, com, bon = m.verify_step(ids, torch.from_numpy(tok).cuda(), q=torch.from_numpy(q).cuda(),
                                      u=torch.from_numpy(u).cuda(), temperature=temp)
        clear = stochastic_margin(p, q, tok[:, 1:], u, n_ref)
        acc, com = acc.cpu().numpy(), com.cpu().numpy()
        for b in range(2):
            if clear[b]:
                compared += 1
                assert acc[b] == n_ref[b]
                np.testing.assert_array_equal(com[b], com_ref[b])
            else:
                near += 1
        o.commit(ids, n_ref, gamma + 1)
        for b in range(2):
            hist[b].extend(int(t) for t in com_ref[b, :n_ref[b] + 1])
        if not ((acc == n_ref).all() and (com == com_ref).all()):
            ids, o = _fresh(w, m, [np.array(h) for h in hist])   # re-sync both sides
        pending = com_ref[np.arange(2), n_ref]
    margins(compared, near)
    assert compared >= 16, (compared, near)


def test_decode_steps_match_oracle(tiny, margins):
    """Twelve teacher-forced decode steps: logits within the tolerance every step and
    the next token equal to the oracle's wherever its top-2 gap is clear.  Both sides
    are fed the oracle's token, so a near-tie step leaves the two caches alike."""
    w, m = tiny
    prompts = _prompts([64, 20], 9)
    ids, o = _fresh(w, m, prompts)
    pending = np.array([p[-1] for p in prompts])
    compared = near = 0
    for step in range(12):
        ref = o.forward(ids, pending[:, None])
        nxt = m.decode_step(ids, torch.from_numpy(pending).cuda()).cpu().numpy()
        got = m.debug_logits(2).cpu().numpy()
        assert rel_err(got, ref[:, 0]) < TOL
        want = ref[:, 0].argmax(-1)
        gap = np.sort(ref[:, 0], -1)
        clear = gap[:, -1] - gap[:, -2] > 1e-2
        assert (nxt[clear] == want[clear]).all()
        compared += int(clear.sum())
        near += int((~clear).sum())
        o.commit(ids, [0, 0], 1)
        pending = want
    lens, pt = m.kv_state(ids)
    assert lens == o.lengths(ids).tolist()
    np.testing.assert_array_equal(np.array(pt), o.kv.page_table_array(ids))
    margins(compared, near)
    assert compared >= 20, (compared, near)


def test_sampled_decode_step(tiny):
    w, m = tiny
    prompts = _prompts([40, 41], 12)
    ids, o = _fresh(w, m, prompts)
    pending = np.array([p[-1] for p in prompts])
    u = np.array([0.3, 0.9], np.float32)
    ref = o.forward(ids, pending[:, None])
    p = A.target_probs(ref, 1.0)
    n_ref, com_ref, tok_ref, _ = A.accept_stochastic(p, np.zeros((2, 0, synth.TINY.vocab), np.float32),
                                                     np.zeros((2, 0)), u[:, None])
    nxt = m.decode_step(ids, torch.from_numpy(pending).cuda(), temperature=1.0, u=torch.from_numpy(u).cuda())
    clear = stochastic_margin(p, np.zeros((2, 0, synth.TINY.vocab), np.float32), np.zeros((2, 0)), u[:, None],
                              n_ref)
    got = nxt.cpu().numpy()
    assert (got[clear] == tok_ref[clear]).all()


TREE15 = [-1, 0, 0, 1, 1, 2, 2, 3, 3, 4, 4, 5, 5, 6, 6]    # binary, three levels below the root


def test_tree_verify(tiny, margins):
    """15-node tree, six rounds: ancestor-masked logits, the greedy walk, path KV
    compaction and the page table after rollback of the rejected branches.  A round
    with a near-tie on the walk is counted, and both sides restart from the oracle's
    committed history."""
    w, m = tiny
    prompts = _prompts([100, 70], 13)
    ids, o = _fresh(w, m, prompts)
    hist = [list(map(int, p)) for p in prompts]
    N = len(TREE15)
    rng = np.random.default_rng(14)
    compared = near = 0
    for r in range(6):
        tok = np.zeros((2, N), np.int64)
        tok[:, 0] = [h[-1] for h in hist]
        tok[:, 1:] = rng.integers(0, synth.TINY.vocab, (2, N - 1))
        ref = o.forward(ids, tok, parent=np.array(TREE15))
        am = ref.argmax(-1)
        for c in range(1, N):                    # plant matches along some branches
            if rng.random() < 0.6:
                tok[:, c] = am[:, TREE15[c]]
                ref = o.forward(ids, tok, parent=np.array(TREE15))
                am = ref.argmax(-1)
        n_ref, path, com_ref, bon_ref = A.accept_tree_greedy(ref, tok, np.array(TREE15))
        acc, com, bon = m.verify_tree_step(ids, torch.from_numpy(tok).cuda(), TREE15)
        got = m.debug_logits(2 * N).cpu().numpy().reshape(ref.shape)
        assert rel_err(got, ref) < TOL
        gap = np.sort(ref, -1)
        clear = ((gap[..., -1] - gap[..., -2]) > 1e-2).all(axis=1)
        acc, com = acc.cpu().numpy(), com.cpu().numpy()
        for b in range(2):
            if clear[b]:
                compared += 1
                assert acc[b] == n_ref[b]
                np.testing.assert_array_equal(com[b, :n_ref[b] + 1], com_ref[b, :n_ref[b] + 1])
            else:
                near += 1
        for b in range(2):
            hist[b].extend(int(t) for t in com_ref[b, :n_ref[b] + 1])
        if not clear.all():                      # the GPU may have walked elsewhere: restart both
            ids, o = _fresh(w, m, [np.array(h) for h in hist])
            continue
        L0 = o.lengths(ids)
        o.commit_tree(ids, path)
        lens, pt = m.kv_state(ids)
        assert lens == o.lengths(ids).tolist()
        np.testing.assert_array_equal(np.array(pt), o.kv.page_table_array(ids))
        for b, s in enumerate(ids):              # compacted path KV, layer 0 and last
            for layer in (0, synth.TINY.n_layers - 1):
                k, v = m.read_kv(layer, s, int(L0[b]), int(n_ref[b]) + 1)
                kr = np.stack([o.kv.k[layer, o.kv.slot(s, t)[0], :, o.kv.slot(s, t)[1]]
                               for t in range(int(L0[b]), int(L0[b]) + int(n_ref[b]) + 1)])
                assert rel_err(k.float().numpy(), kr) < TOL
    margins(compared, near)
    assert compared >= 6, (compared, near)


def test_capacity_error_is_reported(tiny):
    need_gpu()
    from speculative_decoding_verify_step_gb300 import spec
    w, _ = tiny
    m = cuda_model(synth.TINY, w, max_batch=2, max_width=4, max_seq_len=128, num_pages=3)
    try:
        m.seq_reset([0, 1])
        m.prefill([0], torch.zeros(1, 100, dtype=torch.int32).cuda(), [100])   # 99 cached: 2 pages
        m.sync_status()
        m.prefill([1], torch.zeros(1, 80, dtype=torch.int32).cuda(), [80])     # needs 2, 1 left
        with pytest.raises(spec.SpecError) as e:
            m.sync_status()
        assert e.value.status == 4
        m.sync_status()                          # cleared; the context is still usable
        m.seq_reset([1])
        m.prefill([1], torch.zeros(1, 10, dtype=torch.int32).cuda(), [10])
        m.sync_status()
    finally:
        m.close()


def test_timeout_status_is_reported(tiny):
    """A bounded device wait that nothing completes runs out (~1 ms here), records
    SPEC_ERR_TIMEOUT for the host, and leaves the context usable."""
    need_gpu()
    from speculative_decoding_verify_step_gb300 import spec
    w, _ = tiny
    m = cuda_model(synth.TINY, w, max_batch=2, max_width=4, max_seq_len=128, num_pages=8)
    try:
        m.sync_status()
        m.debug_wait_probe(2_000_000)
        with pytest.raises(spec.SpecError) as e:
            m.sync_status()
        assert e.value.status == 6
        m.sync_status()                          # cleared
        m.seq_reset([0])
        m.prefill([0], torch.zeros(1, 10, dtype=torch.int32).cuda(), [10])
        m.sync_status()
        with pytest.raises(spec.SpecError):
            m.debug_wait_probe(0)                # budget out of range: refused on the host
    finally:
        m.close()


def test_invalid_arguments(tiny):
    need_gpu()
    from speculative_decoding_verify_step_gb300 import spec
    w, m = tiny
    tok = torch.zeros(2, 4, dtype=torch.int32).cuda()
    with pytest.raises(spec.SpecError) as e:       # sampled without q/u: never a greedy fallback
        m.verify_step([0, 1], tok, temperature=1.0)
    assert e.value.status == 1
    with pytest.raises(spec.SpecError):
        m.verify_step(list(range(5)), torch.zeros(5, 4, dtype=torch.int32).cuda())
    with pytest.raises(spec.SpecError):
        m.verify_step([0, 1], torch.zeros(2, 17, dtype=torch.int32).cuda())
    with pytest.raises(spec.SpecError):
        m.verify_tree_step([0, 1], tok, [-1, 0, 2, 1])
    bad = torch.full((2, 4), 5000, dtype=torch.int32).cuda()
    m.seq_reset([0, 1])
    m.prefill([0, 1], torch.zeros(2, 8, dtype=torch.int32).cuda(), [8, 8])
    m.verify_step([0, 1], bad)
    with pytest.raises(spec.SpecError) as e:
        m.sync_status()
    assert e.value.status == 1


def test_repeated_sequence_ids_are_refused(tiny):
    """One sequence named twice in a call would have two windows write its slots and
    race on its length: the call is refused on the device (SPEC_ERR_INVALID_ARG) and
    no sequence's length or pages change."""
    need_gpu()
    from speculative_decoding_verify_step_gb300 import spec
    w, m = tiny
    m.seq_reset([0, 1, 2, 3])
    m.prefill([0, 1], torch.zeros(2, 63, dtype=torch.int32).cuda(), [63, 40])   # seq 0: 62 cached
    m.sync_status()
    before = m.kv_state([0, 1])
    for ids in ([0, 0], [1, 0, 1]):
        tok = torch.ones(len(ids), 4, dtype=torch.int32).cuda()
        m.verify_step(ids, tok)                      # window would cross seq 0's page boundary
        with pytest.raises(spec.SpecError) as e:
            m.sync_status()
        assert e.value.status == 1
        assert m.kv_state([0, 1]) == before
    m.verify_step([0, 1], torch.ones(2, 4, dtype=torch.int32).cuda())   # distinct ids still work
    m.sync_status()
    lens, _ = m.kv_state([0, 1])
    assert lens[0] > before[0][0] and lens[1] > before[0][1]


def test_verify_round_on_an_exhausted_pool_keeps_the_length(tiny):
    """A sequence whose window cannot get its pages keeps its length and page table
    (the round's other sequences commit); once pages are free again it continues."""
    need_gpu()
    from speculative_decoding_verify_step_gb300 import spec
    w, _ = tiny
    m = cuda_model(synth.TINY, w, max_batch=3, max_width=8, max_seq_len=256, num_pages=3)
    try:
        m.seq_reset([0, 1, 2])
        m.prefill([0, 1], torch.zeros(2, 65, dtype=torch.int32).cuda(), [65, 64])  # 64 and 63 cached: pages 0, 1
        m.prefill([2], torch.zeros(1, 30, dtype=torch.int32).cuda(), [30])         # page 2: the pool is full
        m.sync_status()
        before = m.kv_state([0, 1, 2])
        tok = torch.ones(3, 8, dtype=torch.int32).cuda()
        acc, _, _ = m.verify_step([2, 1, 0], tok)    # seq 2 fits its page; 1 and 0 need a second one
        with pytest.raises(spec.SpecError) as e:
            m.sync_status()
        assert e.value.status == 4
        lens, pt = m.kv_state([0, 1, 2])
        assert lens[:2] == before[0][:2] and pt[:2] == before[1][:2]
        assert lens[2] == before[0][2] + 1 + int(acc[0])
        m.seq_reset([2])                              # page 2 back to the pool
        m.verify_step([0], tok[:1])                   # slots 64..71: the length passes 64, page 2 stays
        m.sync_status()
        lens, pt = m.kv_state([0])
        assert lens[0] > before[0][0] and pt[0][:2] == [0, 2]
    finally:
        m.close()


def test_first_error_of_a_round_is_reported_in_batch_order(tiny):
    """Two device-side errors in one round: the status word keeps the first in batch
    order -- a sequence that cannot get its page (SPEC_ERR_CAPACITY) listed before a
    sequence whose verify length exceeds the width (SPEC_ERR_INVALID_ARG), and the
    other way round; the sequence without its page keeps its length either way."""
    need_gpu()
    from speculative_decoding_verify_step_gb300 import spec
    w, _ = tiny
    m = cuda_model(synth.TINY, w, max_batch=3, max_width=8, max_seq_len=256, num_pages=3)
    try:
        m.seq_reset([0, 1, 2])
        m.prefill([0, 1], torch.zeros(2, 65, dtype=torch.int32).cuda(), [65, 64])  # 64 and 63 cached: pages 0, 1
        m.prefill([2], torch.zeros(1, 30, dtype=torch.int32).cuda(), [30])         # page 2: the pool is full
        m.sync_status()
        before = m.kv_state([0])
        tok = torch.ones(14, dtype=torch.int32).cuda()  # 5 + 9 rows, packed
        # sequence 0 needs a second page (64 + 5 slots); sequence 2 asks for 9 rows of 8
        for ids, lens, first in (([0, 2], [5, 9], 4), ([2, 0], [9, 5], 1)):
            m.verify_ragged(ids, tok, lens, spec.RAGGED_COMPACT, gamma=7)
            with pytest.raises(spec.SpecError) as e:
                m.sync_status()
            assert e.value.status == first, (ids, lens)
            assert m.kv_state([0]) == before
    finally:
        m.close()


def test_kv_write_gives_a_sequence_the_callers_cache(tiny):
    """spec_kv_write: the values read back bit for bit, pages taken lowest first, the
    length set; an exhausted pool reports SPEC_ERR_CAPACITY; wrong shapes are refused."""
    need_gpu()
    from speculative_decoding_verify_step_gb300 import spec
    w, _ = tiny
    dims = synth.TINY
    m = cuda_model(dims, w, max_batch=2, max_width=4, max_seq_len=256, num_pages=5)
    try:
        m.seq_reset([0, 1])
        shape = (dims.n_layers, 130, dims.n_kv_heads, dims.head_dim)
        k = synth.normal_fill(shape, seed=1, std=1.0, dtype=torch.float16)
        v = synth.normal_fill(shape, seed=2, std=1.0, dtype=torch.float16)
        m.kv_write(1, k, v)
        m.sync_status()
        lens, pt = m.kv_state([1])
        assert lens == [130] and pt[0][:3] == [0, 1, 2] and pt[0][3] == -1
        for layer in range(dims.n_layers):
            kr, vr = m.read_kv(layer, 1, 0, 130)
            assert torch.equal(kr, k[layer]) and torch.equal(vr, v[layer])
        m.kv_write(0, k[:, :100], v[:, :100])      # needs 2 pages, 2 left
        m.sync_status()
        assert m.kv_state([0])[1][0][:2] == [3, 4]
        m.kv_write(0, k[:, :129], v[:, :129])      # 3 pages: one short after its own 2 return
        with pytest.raises(spec.SpecError) as e:
            m.sync_status()
        assert e.value.status == 4
        lens, pt = m.kv_state([0])
        assert lens == [0] and pt[0][0] == -1           # the pages it took went back to the pool
        m.kv_write(0, k[:, :100], v[:, :100])
        m.sync_status()
        assert m.kv_state([0])[1][0][:2] == [3, 4]
        with pytest.raises(ValueError):
            m.kv_write(0, k[:1], v[:1])            # wrong layer count
    finally:
        m.close()


def test_long_context_attention_matches_oracle():
    """A 4200-token cache: 66 pages per sequence, 5 per CTA of the 16-CTA cluster,
    so the attention splits each page's keys over four warps and combines their
    partials; logits of a verify window and of a decode step match the oracle."""
    need_gpu()
    w = synth.make_weights(synth.TINY, seed=8, gain_jitter=0.1)
    kw = dict(max_batch=2, max_width=8, max_seq_len=4400, num_pages=80)
    m = cuda_model(synth.TINY, w, **kw)
    try:
        g = np.random.default_rng(8)
        prompt = g.integers(0, synth.TINY.vocab, 4200)
        m.seq_reset([0])
        m.prefill([0], torch.from_numpy(prompt[None]).int().cuda(), [4200])
        o = oracle_for(synth.TINY, w, **kw)
        o.prefill([0], [prompt])
        win = np.concatenate([[prompt[-1]], g.integers(0, synth.TINY.vocab, 3)])[None]
        got = m.score([0], torch.from_numpy(win).cuda()).cpu().numpy()
        assert rel_err(got, o.forward([0], win)) < TOL
        m.decode_step([0], torch.from_numpy(win[:, 0]).int().cuda())
        got1 = m.debug_logits(1).cpu().numpy()
        assert rel_err(got1, o.forward([0], win[:, :1])[:, 0]) < TOL
        m.sync_status()
    finally:
        m.close()


@pytest.mark.parametrize("W", [3, 4])
def test_many_sequences_single_cta_attention(W):
    """40 sequences x 4 kv heads leave one CTA per (sequence, kv head) in one wave
    (no cluster merge): logits and the written KV still match the oracle.  At width
    4 the 160 rows take two tcgen05 token tiles (128 + a ragged 32)."""
    need_gpu()
    w = synth.make_weights(synth.TINY, seed=9, gain_jitter=0.1)
    B = 40
    kw = dict(max_batch=B, max_width=4, max_seq_len=128, num_pages=2 * B + 8)
    m = cuda_model(synth.TINY, w, **kw)
    try:
        g = np.random.default_rng(9)
        lens = g.integers(5, 90, B)
        prompts = [g.integers(0, synth.TINY.vocab, n) for n in lens]
        ids = list(range(B))
        m.seq_reset(ids)
        tok = torch.zeros(B, int(lens.max()), dtype=torch.int32)
        for b, pr in enumerate(prompts):
            tok[b, :len(pr)] = torch.as_tensor(pr)
        m.prefill(ids, tok.cuda(), lens.tolist())
        o = oracle_for(synth.TINY, w, **kw)
        o.prefill(ids, prompts)
        win = np.concatenate([np.array([[pr[-1]] for pr in prompts]), g.integers(0, synth.TINY.vocab, (B, W - 1))], 1)
        got = m.score(ids, torch.from_numpy(win).cuda()).cpu().numpy()
        assert rel_err(got, o.forward(ids, win)) < TOL
        lens_m, pt = m.kv_state(ids)
        assert lens_m == o.lengths(ids).tolist()
        m.sync_status()
    finally:
        m.close()
