"""Llama-style target decoder over a paged KV cache (oracle; test infrastructure only).

What the verify forward computes: one target forward pass that scores the
pending token plus gamma drafts per sequence, all W = gamma + 1 rows at once
(Lecture 6 "Optimizing Autoregressive Decode" section 6.1: the target computes
p_1..p_{gamma+1} in a single forward, like a prefill of the block).  Linear
layers act on the flattened rows; attention is done per sequence against that
sequence's own cache (section 4.2, selective batching).

The KV cache keeps the pending-token invariant of section 6.2: it holds the
committed sequence minus its last token; a round writes the window's KV at
slots L..L+W-1 and the commit sets the length to (new committed length - 1),
so rollback is a length edit.  With paged KV, rollback edits the block-table
length and frees the trailing blocks (section 11).  Pages hold 64 tokens, the
page size the ninfer draft-depth sweep pins ("kPagedKVPageSize = 64").

The decoder itself is never printed on the pages; the model is the standard
Llama form the workload names (RMSNorm, RoPE, grouped-query attention, SwiGLU,
untied embedding and LM head).  Readings where the pages are silent:
* RMSNorm: x / sqrt(mean(x^2) + eps) * g.
* RoPE: half-split pairs (i, i + hd/2), inverse frequency theta^(-2i/hd),
  position = absolute token index (tree nodes: L + depth); cos/sin in float64.
* Attention scale 1/sqrt(hd); query head h reads kv head h // (H_q / H_kv).
* Tree window: node j's KV sits in slot L + j; node j sees the cached slots
  < L and the window slots of its ancestors (itself included).  A chain is
  the tree whose parent[j] = j - 1, so one masked attention covers both.
* Arithmetic is float64 on the bf16-rounded weights; activations are not
  rounded to bf16 between steps.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional

import numpy as np

from .accept import tree_ancestors, tree_depths

PAGE = 64


class CapacityError(RuntimeError):
    """No free KV page left."""


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64, exactly; other dtypes are cast."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def weights_to_numpy(weights) -> Dict[str, np.ndarray]:
    """torch weights (bf16 matrices, fp32 gains) -> numpy: uint16 bit patterns / float64."""
    import torch
    out = {}
    for k, t in weights.items():
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            out[k] = t.view(torch.int16).numpy().view(np.uint16)
        else:
            out[k] = t.to(torch.float64).numpy()
    return out


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotary embedding, half-split pairing.  x [..., n_heads, hd], pos [...] (ints).

    Pair (x_i, x_{i+hd/2}) is rotated by angle pos * theta^(-2i/hd):
    (a, b) -> (a cos - b sin, a sin + b cos).
    """
    hd = x.shape[-1]
    half = hd // 2
    inv = np.array([theta ** (-2.0 * i / hd) for i in range(half)], dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv           # [..., half]
    c = np.cos(ang)[..., None, :]
    s = np.sin(ang)[..., None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, visible: np.ndarray) -> np.ndarray:
    """Masked softmax attention with grouped KV heads.

    q [R, Hq, hd], K and V [T, Hk, hd], visible [R, T] bool.  Query head h reads
    kv head h // (Hq / Hk); scores are q.k / sqrt(hd); masked keys get zero weight.
    """
    R, Hq, hd = q.shape
    Hk = K.shape[1]
    grp = Hq // Hk
    out = np.zeros((R, Hq, hd))
    for hq in range(Hq):
        kh = hq // grp
        sc = (q[:, hq] @ K[:, kh].T) / math.sqrt(hd)              # [R, T]
        sc = np.where(visible, sc, -np.inf)
        sc = sc - sc.max(axis=1, keepdims=True)
        e = np.exp(sc)
        pr = e / e.sum(axis=1, keepdims=True)
        out[:, hq] = pr @ V[:, kh]
    return out


class PagedKV:
    """Per-sequence paged KV store with a lowest-free-index-first page allocator."""

    def __init__(self, n_layers, num_pages, n_kv, hd, max_batch, max_pages_per_seq):
        self.num_pages = num_pages
        self.max_pages_per_seq = max_pages_per_seq
        self.k = np.zeros((n_layers, num_pages, n_kv, PAGE, hd), dtype=np.float64)
        self.v = np.zeros_like(self.k)
        self.free = [True] * num_pages
        self.table: List[List[int]] = [[] for _ in range(max_batch)]
        self.length = [0] * max_batch

    def reset(self, s: int):
        for pg in self.table[s]:
            self.free[pg] = True
        self.table[s] = []
        self.length[s] = 0

    def ensure(self, s: int, upto: int):
        """Give sequence s pages covering token slots [0, upto)."""
        need = -(-upto // PAGE)
        if need > self.max_pages_per_seq:
            raise CapacityError(f"sequence {s} needs {need} pages > {self.max_pages_per_seq}")
        while len(self.table[s]) < need:
            try:
                pg = self.free.index(True)
            except ValueError:
                raise CapacityError("KV page pool exhausted") from None
            self.free[pg] = False
            self.table[s].append(pg)

    def truncate(self, s: int, new_len: int):
        """Set the length and free every page whose first slot is >= new_len."""
        keep = -(-new_len // PAGE)
        for pg in self.table[s][keep:]:
            self.free[pg] = True
        self.table[s] = self.table[s][:keep]
        self.length[s] = new_len

    def slot(self, s: int, t: int):
        return self.table[s][t // PAGE], t % PAGE

    def page_table_array(self, seq_ids) -> np.ndarray:
        out = np.full((len(seq_ids), self.max_pages_per_seq), -1, dtype=np.int64)
        for i, s in enumerate(seq_ids):
            out[i, :len(self.table[s])] = self.table[s]
        return out


class OracleDecoder:
    """The target model of the verify round, with its own KV cache."""

    def __init__(self, dims, weights: Dict[str, object], *, max_batch: int,
                 max_seq_len: int, num_pages: int):
        self.dims = dims
        self.max_batch = max_batch
        self.max_seq_len = max_seq_len
        self._w = weights             # numpy: uint16 bf16 bit patterns, float gains
        self._cache: Dict[str, np.ndarray] = {}
        self.kv = PagedKV(dims.n_layers, num_pages, dims.n_kv_heads, dims.head_dim,
                          max_batch, -(-max_seq_len // PAGE))
        self.keep_f64 = True          # cache float64 copies of the weights

    # ------------------------------------------------------------------ weights
    def w(self, name: str) -> np.ndarray:
        """Weight `name` as float64 (bf16 matrices are widened exactly)."""
        if name in self._cache:
            return self._cache[name]
        f = bf16_bits_to_f64(self._w[name])
        if self.keep_f64:
            self._cache[name] = f
        return f

    def embed_rows(self, tokens: np.ndarray) -> np.ndarray:
        t = np.asarray(tokens, dtype=np.int64)
        return bf16_bits_to_f64(self._w["embed"][t.reshape(-1)]).reshape(*t.shape, self.dims.d_model)

    # ---------------------------------------------------------------- sequences
    def reset(self, seq_ids):
        for s in seq_ids:
            self.kv.reset(int(s))

    def lengths(self, seq_ids) -> np.ndarray:
        return np.array([self.kv.length[int(s)] for s in seq_ids], dtype=np.int64)

    # ------------------------------------------------------------------ forward
    def forward(self, seq_ids, tokens, parent: Optional[np.ndarray] = None,
                want_logits: bool = True, return_hidden: bool = False):
        """Score a window of W rows per sequence; writes the window's KV at slots
        L..L+W-1 but leaves the committed lengths unchanged.

        tokens [B, W] ints; parent [W] (tree, parent[0] = -1) or None (chain).
        Returns logits [B, W, V] float64 (and the final-normed hidden [B, W, d]).
        """
        dims = self.dims
        tokens = np.asarray(tokens, dtype=np.int64)
        B, W = tokens.shape
        if parent is None:
            parent = np.arange(-1, W - 1, dtype=np.int64)
        parent = np.asarray(parent, dtype=np.int64)
        depth = tree_depths(parent)
        anc = tree_ancestors(parent)
        seq_ids = [int(s) for s in seq_ids]
        L = [self.kv.length[s] for s in seq_ids]
        for b, s in enumerate(seq_ids):                 # allocation order: b = 0..B-1
            if L[b] + W > self.max_seq_len:
                raise CapacityError(f"sequence {s}: {L[b]} + {W} > max_seq_len")
            self.kv.ensure(s, L[b] + W)
        pos = np.array([[L[b] + depth[j] for j in range(W)] for b in range(B)])

        Hq, Hk, hd = dims.n_heads, dims.n_kv_heads, dims.head_dim
        h = self.embed_rows(tokens)                     # [B, W, d] residual stream
        for li in range(dims.n_layers):
            p = f"layers.{li}."
            a = rmsnorm(h, self.w(p + "attn_norm"), dims.rms_eps)
            q = (a @ self.w(p + "wq").T).reshape(B, W, Hq, hd)
            k = (a @ self.w(p + "wk").T).reshape(B, W, Hk, hd)
            v = (a @ self.w(p + "wv").T).reshape(B, W, Hk, hd)
            q = rope(q, pos, dims.rope_theta)
            k = rope(k, pos, dims.rope_theta)
            o = np.zeros((B, W, Hq, hd))
            for b, s in enumerate(seq_ids):
                for j in range(W):                      # window KV at slot L + j
                    pg, off = self.kv.slot(s, L[b] + j)
                    self.kv.k[li, pg, :, off] = k[b, j]
                    self.kv.v[li, pg, :, off] = v[b, j]
                n_keys = L[b] + W
                K = np.empty((n_keys, Hk, hd))
                Vv = np.empty((n_keys, Hk, hd))
                for t in range(n_keys):
                    pg, off = self.kv.slot(s, t)
                    K[t] = self.kv.k[li, pg, :, off]
                    Vv[t] = self.kv.v[li, pg, :, off]
                visible = np.zeros((W, n_keys), dtype=bool)
                visible[:, :L[b]] = True
                for j in range(W):
                    for i in anc[j]:
                        visible[j, L[b] + i] = True
                o[b] = attention(q[b], K, Vv, visible)
            h = h + o.reshape(B, W, Hq * hd) @ self.w(p + "wo").T
            f = rmsnorm(h, self.w(p + "ffn_norm"), dims.rms_eps)
            gate = f @ self.w(p + "w_gate").T
            up = f @ self.w(p + "w_up").T
            h = h + (silu(gate) * up) @ self.w(p + "w_down").T
        hid = rmsnorm(h, self.w("final_norm"), dims.rms_eps)
        logits = hid @ self.w("lm_head").T if want_logits else None
        if return_hidden:
            return logits, hid
        return logits

    def load_cache(self, s: int, k: np.ndarray, v: np.ndarray):
        """Start sequence s from a given cache: k, v [n_layers, n, n_kv, hd] become
        its KV at slots 0..n-1 (pages taken lowest free first) and its length n.
        The GPU path's counterpart receives the same values, so both sides attend
        over one cache without a prefill."""
        s = int(s)
        n = int(k.shape[1])
        self.kv.reset(s)
        self.kv.ensure(s, n)
        for t in range(n):
            pg, off = self.kv.slot(s, t)
            self.kv.k[:, pg, :, off] = k[:, t]
            self.kv.v[:, pg, :, off] = v[:, t]
        self.kv.truncate(s, n)

    # ------------------------------------------------------------------- rounds
    def prefill(self, seq_ids, prompts):
        """Write KV for prompt[:-1] of each sequence (lengths may differ); the last
        prompt token becomes the pending token.  prompts: list of 1-D int arrays."""
        for s, pr in zip(seq_ids, prompts):
            pr = np.asarray(pr, dtype=np.int64)
            assert len(pr) >= 1
            if len(pr) > 1:
                self.forward([s], pr[None, :-1], want_logits=False)
                self.kv.truncate(int(s), self.kv.length[int(s)] + len(pr) - 1)

    def commit(self, seq_ids, accepted, width: int):
        """Chain commit: L <- L + 1 + n; free pages wholly beyond the new length."""
        for s, n in zip(seq_ids, accepted):
            s = int(s)
            assert 0 <= int(n) < width
            self.kv.truncate(s, self.kv.length[s] + 1 + int(n))

    def commit_tree(self, seq_ids, path):
        """Tree commit: move the accepted path's KV (nodes at depths 1..n, all layers)
        into slots L+1..L+n, then truncate to L + 1 + n."""
        for b, s in enumerate(seq_ids):
            s = int(s)
            L = self.kv.length[s]
            nodes = [int(c) for c in path[b] if c >= 0]
            for d, c in enumerate(nodes, start=1):
                src = self.kv.slot(s, L + c)
                dst = self.kv.slot(s, L + d)
                self.kv.k[:, dst[0], :, dst[1]] = self.kv.k[:, src[0], :, src[1]].copy()
                self.kv.v[:, dst[0], :, dst[1]] = self.kv.v[:, src[0], :, src[1]].copy()
            self.kv.truncate(s, L + 1 + len(nodes))
