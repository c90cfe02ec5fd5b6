"""Thin Python binding of the verify-round C ABI (include/spec_verify.h).

Argument marshalling only: every step of the round runs in the CUDA library.
Tensors are torch CUDA tensors (device memory and streams come from PyTorch);
the current torch stream is passed to every call.  Loading fails loudly when
the library has not been built -- there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, Optional, Sequence, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

SPEC_OK = 0
STATUS_NAMES = {0: "SPEC_OK", 1: "SPEC_ERR_INVALID_ARG", 2: "SPEC_ERR_UNSUPPORTED_DEVICE", 3: "SPEC_ERR_OOM",
                4: "SPEC_ERR_CAPACITY", 5: "SPEC_ERR_CUDA", 6: "SPEC_ERR_TIMEOUT", 7: "SPEC_ERR_UNSUPPORTED"}

WEIGHT_KIND = {"embed": 0, "lm_head": 1, "final_norm": 2, "attn_norm": 3, "wq": 4, "wk": 5, "wv": 6, "wo": 7,
               "ffn_norm": 8, "w_gate": 9, "w_up": 10, "w_down": 11}


class SpecError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class spec_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn_dim", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("page_size", ctypes.c_int32), ("max_batch", ctypes.c_int32), ("max_width", ctypes.c_int32),
                ("max_seq_len", ctypes.c_int32), ("num_pages", ctypes.c_int32)]


EXPORTS = ["spec_model_create", "spec_model_destroy", "spec_model_set_weight", "spec_seq_reset", "spec_prefill",
           "spec_decode_step", "spec_verify_step", "spec_verify_tree_step", "spec_score", "spec_accept_probs",
           "spec_accept_greedy", "spec_get_kv_state", "spec_read_kv", "spec_debug_logits", "spec_debug_wait_probe",
           "spec_kv_fill_random", "spec_sync_status", "spec_max_pages_per_seq", "spec_last_launch_count", "spec_last_error",
           "spec_set_profiling", "spec_read_profile", "spec_accept_greedy_noalloc", "spec_verify_ragged",
           "spec_adjust_probs", "spec_verify_tree_sampled", "spec_accept_tree_probs", "spec_kv_write"]

RAGGED_CAP_ACCEPT, RAGGED_COMPACT = 1, 2

PROFILE_CLASSES = ["qkv", "o", "gate_up", "down", "lm_head", "attention"]

_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (raises if it is missing: build it with __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build the CUDA library first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P, I32, I64, F32, U64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_uint64
    sig = {
        "spec_model_create": (I32, [ctypes.POINTER(spec_config), ctypes.POINTER(P)]),
        "spec_model_destroy": (None, [P]),
        "spec_model_set_weight": (I32, [P, I32, I32, P, I64, P]),
        "spec_seq_reset": (I32, [P, I32, P, P]),
        "spec_prefill": (I32, [P, I32, P, P, I32, P, P]),
        "spec_decode_step": (I32, [P, I32, P, P, F32, P, P, P, P, P]),
        "spec_verify_step": (I32, [P, I32, I32, P, P, P, P, F32, P, P, P, P, P, P]),
        "spec_verify_tree_step": (I32, [P, I32, I32, P, P, P, P, P, P, P]),
        "spec_verify_ragged": (I32, [P, I32, I32, P, P, P, I32, I32, P, P, F32, P, P, P, P, P, P]),
        "spec_adjust_probs": (I32, [I32, I32, P, P, P, P, I32, P]),
        "spec_verify_tree_sampled": (I32, [P, I32, I32, P, P, P, P, P, F32, P, P, P, P, P, P]),
        "spec_accept_tree_probs": (I32, [I32, I32, I32, P, P, P, P, P, P, P, P, P]),
        "spec_score": (I32, [P, I32, I32, P, P, P, P, P]),
        "spec_accept_probs": (I32, [I32, I32, I32, P, P, P, P, P, P, P, P]),
        "spec_accept_greedy": (I32, [I32, I32, I32, P, P, P, P, P, P]),
        "spec_get_kv_state": (I32, [P, I32, P, P, P]),
        "spec_read_kv": (I32, [P, I32, I32, I32, I32, P, P]),
        "spec_debug_logits": (I32, [P, P, I64, P]),
        "spec_debug_wait_probe": (I32, [P, I64, P]),
        "spec_kv_fill_random": (I32, [P, I32, P, P, U64, F32, P]),
        "spec_kv_write": (I32, [P, I32, I32, P, P, P]),
        "spec_sync_status": (I32, [P, P]),
        "spec_max_pages_per_seq": (I32, [P]),
        "spec_last_launch_count": (I32, [P]),
        "spec_last_error": (ctypes.c_char_p, []),
        "spec_set_profiling": (I32, [P, I32]),
        "spec_accept_greedy_noalloc": (I32, [I32, I32, I32, P, P, P, P, P, P]),
        "spec_read_profile": (I32, [P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != SPEC_OK:
        raise SpecError(status, _lib.spec_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    assert t.is_contiguous(), "tensors must be contiguous"
    return ctypes.c_void_p(t.data_ptr())


def _i32_host(xs: Sequence[int]):
    arr = (ctypes.c_int32 * len(xs))(*[int(x) for x in xs])
    return arr


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dev_i32(t, device) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        t = torch.as_tensor(t)
    return t.to(device=device, dtype=torch.int32).contiguous()


def _f32(t: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    """q and u are fp32 on the C side: convert (no copy when already fp32 and contiguous)."""
    return None if t is None else t.to(dtype=torch.float32).contiguous()


def _opt_dev(t, device, dtype):
    """None stays None (setting off); a list, array or tensor becomes a device tensor."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        t = torch.as_tensor(t)
    return t.to(device=device, dtype=dtype).contiguous()


class SpecModel:
    """Owns one spec_model handle.  Method names follow the C ABI without the prefix."""

    def __init__(self, dims, *, max_batch: int, max_width: int, max_seq_len: int, num_pages: int):
        lib = load_library()
        self.dims = dims
        cfg = spec_config(dims.n_layers, dims.d_model, dims.n_heads, dims.n_kv_heads, dims.head_dim, dims.ffn_dim,
                          dims.vocab, dims.rms_eps, dims.rope_theta, 64, max_batch, max_width, max_seq_len, num_pages)
        self.cfg = cfg
        h = ctypes.c_void_p()
        _check(lib.spec_model_create(ctypes.byref(cfg), ctypes.byref(h)))
        self.handle = h
        self.device = torch.device("cuda", torch.cuda.current_device())
        self.max_pages = lib.spec_max_pages_per_seq(h)

    def close(self):
        if getattr(self, "handle", None):
            _lib.spec_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---------------------------------------------------------------- weights
    def set_weight(self, name: str, tensor: torch.Tensor):
        """name: synth-style ('embed', 'layers.3.wq', ...).  bf16 matrices / fp32 gains."""
        parts = name.split(".")
        layer, kind = (int(parts[1]), parts[2]) if parts[0] == "layers" else (0, parts[0])
        want = torch.float32 if kind.endswith("norm") else torch.bfloat16
        t = tensor.to(want).contiguous()
        _check(_lib.spec_model_set_weight(self.handle, WEIGHT_KIND[kind], layer, _ptr(t), t.numel(), _stream()))
        torch.cuda.current_stream().synchronize()  # `t` may be a temporary

    def load_weights(self, items: Iterable[Tuple[str, torch.Tensor]]):
        for name, t in items:
            self.set_weight(name, t)

    # -------------------------------------------------------------- sequences
    def seq_reset(self, seq_ids: Sequence[int]):
        ids = _i32_host(seq_ids)
        _check(_lib.spec_seq_reset(self.handle, len(seq_ids), ids, _stream()))

    def prefill(self, seq_ids, tokens: torch.Tensor, lens: Sequence[int]):
        sid = _dev_i32(seq_ids, self.device)
        tok = _dev_i32(tokens, self.device)
        _check(_lib.spec_prefill(self.handle, sid.numel(), _ptr(sid), _ptr(tok), tok.shape[1], _i32_host(lens),
                                 _stream()))
        torch.cuda.current_stream().synchronize()

    def decode_step(self, seq_ids, tok, temperature: float = 0.0, u=None, out=None, top_k=None, top_p=None):
        sid = _dev_i32(seq_ids, self.device)
        tk = _dev_i32(tok, self.device)
        B = sid.numel()
        out = torch.empty(B, dtype=torch.int32, device=self.device) if out is None else out
        kk, pp = _opt_dev(top_k, self.device, torch.int32), _opt_dev(top_p, self.device, torch.float32)
        u = _f32(u)
        _check(_lib.spec_decode_step(self.handle, B, _ptr(sid), _ptr(tk), float(temperature), _ptr(kk), _ptr(pp),
                                     _ptr(u), _ptr(out), _stream()))
        return out

    def verify_step(self, seq_ids, tok, q=None, u=None, temperature: float = 0.0, outs=None, top_k=None,
                    top_p=None):
        """tok [B, gamma+1] (pending + drafts).  Returns (accepted [B], committed [B, W], bonus [B]).
        top_k / top_p: per-sequence sampling adjustments of sampled rounds (None = off)."""
        sid = _dev_i32(seq_ids, self.device)
        tk = _dev_i32(tok, self.device)
        B, W = tk.shape
        if outs is None:
            outs = (torch.empty(B, dtype=torch.int32, device=self.device),
                    torch.empty(B, W, dtype=torch.int32, device=self.device),
                    torch.empty(B, dtype=torch.int32, device=self.device))
        acc, com, bon = outs
        kk, pp = _opt_dev(top_k, self.device, torch.int32), _opt_dev(top_p, self.device, torch.float32)
        q, u = _f32(q), _f32(u)
        _check(_lib.spec_verify_step(self.handle, B, W - 1, _ptr(sid), _ptr(tk), _ptr(q), _ptr(u),
                                     float(temperature), _ptr(kk), _ptr(pp), _ptr(acc), _ptr(com), _ptr(bon),
                                     _stream()))
        return acc, com, bon

    def verify_ragged(self, seq_ids, tok, verify_lens, mode: int, q=None, u=None, temperature: float = 0.0,
                      gamma: Optional[int] = None, outs=None, top_k=None, top_p=None):
        """mode RAGGED_CAP_ACCEPT: tok [B, gamma+1]; RAGGED_COMPACT: tok packed [sum(verify_lens)].
        verify_lens: per-sequence rows (list or tensor).  Returns (accepted, committed [B, gamma+1], bonus)."""
        sid = _dev_i32(seq_ids, self.device)
        tk = _dev_i32(tok, self.device)
        lens = _dev_i32(verify_lens, self.device)
        B = sid.numel()
        if gamma is None:
            gamma = tk.shape[1] - 1 if mode == RAGGED_CAP_ACCEPT else int(lens.max().item()) - 1
        total = int(tk.numel()) if mode == RAGGED_COMPACT else B * (gamma + 1)
        if outs is None:
            outs = (torch.empty(B, dtype=torch.int32, device=self.device),
                    torch.empty(B, gamma + 1, dtype=torch.int32, device=self.device),
                    torch.empty(B, dtype=torch.int32, device=self.device))
        acc, com, bon = outs
        kk, pp = _opt_dev(top_k, self.device, torch.int32), _opt_dev(top_p, self.device, torch.float32)
        q, u = _f32(q), _f32(u)
        _check(_lib.spec_verify_ragged(self.handle, B, gamma, _ptr(sid), _ptr(tk), _ptr(lens), total, mode, _ptr(q),
                                       _ptr(u), float(temperature), _ptr(kk), _ptr(pp), _ptr(acc), _ptr(com),
                                       _ptr(bon), _stream()))
        return acc, com, bon

    def verify_tree_step(self, seq_ids, tok, parent: Sequence[int], outs=None):
        sid = _dev_i32(seq_ids, self.device)
        tk = _dev_i32(tok, self.device)
        B, N = tk.shape
        if outs is None:
            outs = (torch.empty(B, dtype=torch.int32, device=self.device),
                    torch.empty(B, N, dtype=torch.int32, device=self.device),
                    torch.empty(B, dtype=torch.int32, device=self.device))
        acc, com, bon = outs
        _check(_lib.spec_verify_tree_step(self.handle, B, N, _ptr(sid), _ptr(tk), _i32_host(parent), _ptr(acc),
                                          _ptr(com), _ptr(bon), _stream()))
        return acc, com, bon

    def verify_tree_sampled(self, seq_ids, tok, parent: Sequence[int], u, q=None, temperature: float = 1.0,
                            outs=None, top_k=None, top_p=None):
        """Sampled tree round: u [B, N]; q [B, N, V] (children of node v drawn from q[:, v])
        or None (deterministic candidates).  Returns (accepted, committed [B, N], bonus)."""
        sid = _dev_i32(seq_ids, self.device)
        tk = _dev_i32(tok, self.device)
        B, N = tk.shape
        if outs is None:
            outs = (torch.empty(B, dtype=torch.int32, device=self.device),
                    torch.empty(B, N, dtype=torch.int32, device=self.device),
                    torch.empty(B, dtype=torch.int32, device=self.device))
        acc, com, bon = outs
        kk, pp = _opt_dev(top_k, self.device, torch.int32), _opt_dev(top_p, self.device, torch.float32)
        q, u = _f32(q), _f32(u)
        _check(_lib.spec_verify_tree_sampled(self.handle, B, N, _ptr(sid), _ptr(tk), _i32_host(parent), _ptr(q),
                                             _ptr(u), float(temperature), _ptr(kk), _ptr(pp), _ptr(acc), _ptr(com),
                                             _ptr(bon), _stream()))
        return acc, com, bon

    def score(self, seq_ids, tok, parent: Optional[Sequence[int]] = None, logits_out=None):
        sid = _dev_i32(seq_ids, self.device)
        tk = _dev_i32(tok, self.device)
        B, W = tk.shape
        if logits_out is None:
            logits_out = torch.empty(B, W, self.dims.vocab, dtype=torch.float32, device=self.device)
        _check(_lib.spec_score(self.handle, B, W, _ptr(sid), _ptr(tk), _i32_host(parent) if parent is not None
                               else None, _ptr(logits_out), _stream()))
        return logits_out

    def kv_write(self, seq_id: int, k: torch.Tensor, v: torch.Tensor):
        """Give sequence seq_id the cached K/V k, v: [n_layers, n_tokens, n_kv_heads,
        head_dim] (converted to fp16, the cache's format); its length becomes n_tokens."""
        want = (self.dims.n_layers, k.shape[1], self.dims.n_kv_heads, self.dims.head_dim)
        if tuple(k.shape) != want or tuple(v.shape) != want:
            raise ValueError(f"k, v must be {want}")
        kk = k.to(device=self.device, dtype=torch.float16).contiguous()
        vv = v.to(device=self.device, dtype=torch.float16).contiguous()
        _check(_lib.spec_kv_write(self.handle, int(seq_id), int(k.shape[1]), _ptr(kk), _ptr(vv), _stream()))

    def kv_fill_random(self, seq_ids: Sequence[int], lens: Sequence[int], seed: int = 0, scale: float = 0.5):
        _check(_lib.spec_kv_fill_random(self.handle, len(seq_ids), _i32_host(seq_ids), _i32_host(lens), seed,
                                        scale, _stream()))

    # ------------------------------------------------------------------ state
    def kv_state(self, seq_ids: Sequence[int]):
        n = len(seq_ids)
        lens = (ctypes.c_int32 * n)()
        pt = (ctypes.c_int32 * (n * self.max_pages))()
        _check(_lib.spec_get_kv_state(self.handle, n, _i32_host(seq_ids), lens, pt))
        return list(lens), [list(pt[i * self.max_pages:(i + 1) * self.max_pages]) for i in range(n)]

    def read_kv(self, layer: int, seq_id: int, t0: int, n: int):
        Hkv, hd = self.dims.n_kv_heads, self.dims.head_dim
        k = torch.empty((n, Hkv, hd), dtype=torch.int16)
        v = torch.empty((n, Hkv, hd), dtype=torch.int16)
        _check(_lib.spec_read_kv(self.handle, layer, seq_id, t0, n, ctypes.c_void_p(k.data_ptr()),
                                 ctypes.c_void_p(v.data_ptr())))
        return k.view(torch.float16), v.view(torch.float16)

    def debug_wait_probe(self, budget_cycles: int) -> None:
        """Enqueue one bounded device wait that nothing completes; the next
        sync_status() raises SpecError with SPEC_ERR_TIMEOUT (6)."""
        _check(_lib.spec_debug_wait_probe(self.handle, int(budget_cycles), _stream()))

    def debug_logits(self, rows: int) -> torch.Tensor:
        """Logits of the last forward ([rows, vocab] fp32, device)."""
        out = torch.empty(rows, self.dims.vocab, dtype=torch.float32, device=self.device)
        _check(_lib.spec_debug_logits(self.handle, _ptr(out), out.numel(), _stream()))
        return out

    def sync_status(self):
        _check(_lib.spec_sync_status(self.handle, _stream()))

    def set_profiling(self, enable: bool):
        _check(_lib.spec_set_profiling(self.handle, 1 if enable else 0))

    def read_profile(self):
        """{class: (ms, launches, bytes)} accumulated since the last read."""
        ms = (ctypes.c_double * 6)()
        n = (ctypes.c_int64 * 6)()
        by = (ctypes.c_double * 6)()
        _check(_lib.spec_read_profile(self.handle, ms, n, by))
        return {c: (ms[i], n[i], by[i]) for i, c in enumerate(PROFILE_CLASSES)}

    def last_launch_count(self) -> int:
        return _lib.spec_last_launch_count(self.handle)


# --------------------------------------------------------- standalone acceptance
def spec_accept_probs(p: torch.Tensor, q: Optional[torch.Tensor], x: Optional[torch.Tensor], u: torch.Tensor):
    """p [B, W, V], q [B, W-1, V], x [B, W-1], u [B, W] (CUDA).  Returns (accepted, committed, bonus)."""
    lib = load_library()
    B, W, V = p.shape
    dev = p.device
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    com = torch.empty(B, W, dtype=torch.int32, device=dev)
    bon = torch.empty(B, dtype=torch.int32, device=dev)
    xx = None if x is None else _dev_i32(x, dev)
    pp = p.float().contiguous()
    qq = None if q is None else q.float().contiguous()
    uu = u.float().contiguous()
    _check(lib.spec_accept_probs(B, W - 1, V, _ptr(pp), _ptr(qq), _ptr(xx), _ptr(uu), _ptr(acc), _ptr(com),
                                 _ptr(bon), _stream()))
    torch.cuda.current_stream().synchronize()
    return acc, com, bon


def spec_adjust_probs(p: torch.Tensor, top_k=None, top_p=None, rows_per_setting: int = 1, out=None):
    """Top-k / top-p adjustment of probability rows p [..., V] (CUDA fp32); setting
    i covers rows i*rows_per_setting .. (i+1)*rows_per_setting - 1 of the flattened
    rows.  `out` may be p itself."""
    lib = load_library()
    V = p.shape[-1]
    pp = p.float().contiguous()
    rows = pp.numel() // V
    out = torch.empty_like(pp) if out is None else out
    kk, tp = _opt_dev(top_k, p.device, torch.int32), _opt_dev(top_p, p.device, torch.float32)
    _check(lib.spec_adjust_probs(rows, V, _ptr(pp), _ptr(out), _ptr(kk), _ptr(tp), rows_per_setting, _stream()))
    torch.cuda.current_stream().synchronize()
    return out


def spec_accept_tree_probs(p: torch.Tensor, q: Optional[torch.Tensor], tok, parent: Sequence[int], u: torch.Tensor):
    """p [B, N, V], q [B, N, V] or None, tok [B, N], u [B, N] (CUDA).  Returns (accepted, committed, bonus)."""
    lib = load_library()
    B, N, V = p.shape
    dev = p.device
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    com = torch.empty(B, N, dtype=torch.int32, device=dev)
    bon = torch.empty(B, dtype=torch.int32, device=dev)
    tk = _dev_i32(tok, dev)
    pp = p.float().contiguous()
    qq = None if q is None else q.float().contiguous()
    uu = u.float().contiguous()
    _check(lib.spec_accept_tree_probs(B, N, V, _ptr(pp), _ptr(qq), _ptr(tk), _i32_host(parent), _ptr(uu), _ptr(acc),
                                      _ptr(com), _ptr(bon), _stream()))
    torch.cuda.current_stream().synchronize()
    return acc, com, bon


def spec_accept_greedy_noalloc(logits: torch.Tensor, x: Optional[torch.Tensor], outs=None):
    """Greedy acceptance through the entry point that allocates nothing in the
    library (its scratch is a fixed device array, 4096 rows at most).  `outs`
    lets the caller pass preallocated (accepted, committed, bonus) tensors."""
    lib = load_library()
    B, W, V = logits.shape
    dev = logits.device
    if outs is None:
        outs = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B, W, dtype=torch.int32, device=dev),
                torch.empty(B, dtype=torch.int32, device=dev))
    acc, com, bon = outs
    for t, shape, what in ((acc, (B,), "accepted"), (com, (B, W), "committed"), (bon, (B,), "bonus")):
        if t.dtype != torch.int32 or t.device != dev or tuple(t.shape) != shape:
            raise ValueError(f"{what} must be an int32 tensor of shape {shape} on {dev}")
    xx = None if x is None else _dev_i32(x, dev)
    lg = logits.float().contiguous()
    _check(lib.spec_accept_greedy_noalloc(B, W - 1, V, _ptr(lg), _ptr(xx), _ptr(acc), _ptr(com), _ptr(bon),
                                          _stream()))
    torch.cuda.current_stream().synchronize()
    return acc, com, bon


def spec_accept_greedy(logits: torch.Tensor, x: Optional[torch.Tensor]):
    lib = load_library()
    B, W, V = logits.shape
    dev = logits.device
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    com = torch.empty(B, W, dtype=torch.int32, device=dev)
    bon = torch.empty(B, dtype=torch.int32, device=dev)
    xx = None if x is None else _dev_i32(x, dev)
    lg = logits.float().contiguous()
    _check(lib.spec_accept_greedy(B, W - 1, V, _ptr(lg), _ptr(xx), _ptr(acc), _ptr(com), _ptr(bon), _stream()))
    torch.cuda.current_stream().synchronize()
    return acc, com, bon
