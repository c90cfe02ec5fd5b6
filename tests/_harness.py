"""Test helpers: build oracle decoders from the seeded synthetic weights and run
greedy / speculative loops on them."""
from __future__ import annotations

import dataclasses

import numpy as np

from oracle import accept as A
from oracle.decoder import OracleDecoder, weights_to_numpy
from speculative_decoding_verify_step_gb300 import synth


def oracle_model(dims=synth.TINY, seed=1, gain_jitter=0.0, max_batch=4, max_seq_len=512,
                 num_pages=64, weights=None):
    if weights is None:
        weights = synth.make_weights(dims, seed, gain_jitter=gain_jitter)
    return OracleDecoder(dims, weights_to_numpy(weights), max_batch=max_batch,
                         max_seq_len=max_seq_len, num_pages=num_pages)


def small_dims(**kw):
    """A tiny decoder that is cheap on the CPU; any field can be overridden."""
    base = dict(n_layers=2, d_model=64, n_heads=4, n_kv_heads=2, head_dim=16,
                ffn_dim=96, vocab=50, rms_eps=1e-5, rope_theta=10000.0)
    base.update(kw)
    return synth.Dims(**base)


def greedy_decode(model: OracleDecoder, seq_ids, prompts, steps):
    """Non-speculative greedy generation: one forward of width 1 per token."""
    model.reset(seq_ids)
    model.prefill(seq_ids, prompts)
    pending = np.array([int(p[-1]) for p in prompts])
    out = [[] for _ in seq_ids]
    for _ in range(steps):
        logits = model.forward(seq_ids, pending[:, None])
        nxt = logits[:, 0].argmax(-1)
        model.commit(seq_ids, np.zeros(len(seq_ids), np.int64), 1)
        for b, t in enumerate(nxt):
            out[b].append(int(t))
        pending = nxt
    return out


def greedy_speculative(model: OracleDecoder, seq_ids, prompts, steps, gamma, drafter):
    """Greedy speculative generation; drafter(history_list, gamma) -> gamma tokens."""
    model.reset(seq_ids)
    model.prefill(seq_ids, prompts)
    hist = [list(map(int, p)) for p in prompts]
    out = [[] for _ in seq_ids]
    rounds = 0
    while min(len(o) for o in out) < steps:
        rounds += 1
        toks = np.array([[h[-1]] + list(drafter(h, gamma)) for h in hist])
        logits = model.forward(seq_ids, toks)
        n, committed, _ = A.accept_greedy(logits, toks[:, 1:])
        model.commit(seq_ids, n, gamma + 1)
        for b in range(len(seq_ids)):
            new = [int(t) for t in committed[b, :n[b] + 1]]
            hist[b].extend(new)
            out[b].extend(new)
    return [o[:steps] for o in out], rounds
