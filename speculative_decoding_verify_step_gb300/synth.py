"""Seeded synthetic inputs for the verify round.

This module is the only code shared by the CPU oracle side (tests, the timed CPU
baseline) and the CUDA side (library binding, bench).  It draws random numbers and
nothing else: model weights, prompts, uniforms, Dirichlet(1) draws.  None of the
method's arithmetic (softmax, acceptance, residuals, sampling) lives here.

Workload shapes follow the decoder the verify pages talk about: a Llama-3.1-8B
shaped target (Lecture 6 "Optimizing Autoregressive Decode", section 9.1 uses it
as the target at batch 1, context 1024) and a tiny 2-layer decoder of the same
family for exhaustive checks.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Iterator, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class Dims:
    """Decoder shape.  All projection widths must be multiples of 128."""

    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def with_layers(self, n: int) -> "Dims":
        return dataclasses.replace(self, n_layers=n)


# 2-layer Llama-style decoder: d 256, 4 heads of 64 (MHA), SwiGLU 1024, vocab 1024.
TINY = Dims(n_layers=2, d_model=256, n_heads=4, n_kv_heads=4, head_dim=64,
            ffn_dim=1024, vocab=1024, rms_eps=1e-5, rope_theta=10000.0)

# Llama-3.1-8B shape: 32 layers, d 4096, 32 q / 8 kv heads of 128, ffn 14336, vocab 128256.
LLAMA8B = Dims(n_layers=32, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128,
               ffn_dim=14336, vocab=128256, rms_eps=1e-5, rope_theta=500000.0)


def weight_shapes(dims: Dims) -> Iterator[Tuple[str, Tuple[int, ...], str]]:
    """(name, shape, kind) in generation order; kind is 'matrix' (bf16) or 'gain' (fp32)."""
    d, V = dims.d_model, dims.vocab
    yield "embed", (V, d), "matrix"
    for i in range(dims.n_layers):
        p = f"layers.{i}."
        yield p + "attn_norm", (d,), "gain"
        yield p + "wq", (dims.q_dim, d), "matrix"
        yield p + "wk", (dims.kv_dim, d), "matrix"
        yield p + "wv", (dims.kv_dim, d), "matrix"
        yield p + "wo", (d, dims.q_dim), "matrix"
        yield p + "ffn_norm", (d,), "gain"
        yield p + "w_gate", (dims.ffn_dim, d), "matrix"
        yield p + "w_up", (dims.ffn_dim, d), "matrix"
        yield p + "w_down", (d, dims.ffn_dim), "matrix"
    yield "final_norm", (d,), "gain"
    yield "lm_head", (V, d), "matrix"


def iter_weights(dims: Dims, seed: int, device: str | torch.device = "cpu",
                 std: float = 0.02, gain_jitter: float = 0.0
                 ) -> Iterator[Tuple[str, torch.Tensor]]:
    """Yield (name, tensor) one at a time so 8B-sized models never sit twice in memory.

    Matrices are N(0, std) rounded to bf16 (round-to-nearest-even, torch's cast).
    Norm gains are fp32: 1.0, or 1 + gain_jitter * N(0, 1) when gain_jitter > 0
    (tests use jittered gains so a dropped gain cannot hide).
    """
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    for name, shape, kind in weight_shapes(dims):
        if kind == "matrix":
            t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
            t.mul_(std)
            yield name, t.to(torch.bfloat16)
            del t
        else:
            if gain_jitter > 0:
                t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
                yield name, (1.0 + gain_jitter * t)
            else:
                yield name, torch.ones(shape, device=device, dtype=torch.float32)


def make_weights(dims: Dims, seed: int, device: str | torch.device = "cpu",
                 std: float = 0.02, gain_jitter: float = 0.0) -> Dict[str, torch.Tensor]:
    return dict(iter_weights(dims, seed, device, std, gain_jitter))


def prompts(batch: int, length: int, vocab: int, seed: int) -> torch.Tensor:
    """Random-token prompts [batch, length] int32, uniform over the vocabulary."""
    g = torch.Generator()
    g.manual_seed(seed)
    return torch.randint(0, vocab, (batch, length), generator=g, dtype=torch.int64).to(torch.int32)


def prompt_lengths(batch: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """Per-sequence prompt lengths uniform in [lo, hi] (int32)."""
    g = torch.Generator()
    g.manual_seed(seed)
    return torch.randint(lo, hi + 1, (batch,), generator=g, dtype=torch.int64).to(torch.int32)


def uniforms(shape, seed: int, device: str | torch.device = "cpu") -> torch.Tensor:
    """fp32 uniforms in [0, 1)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32)


def dirichlet1(shape, seed: int, device: str | torch.device = "cpu") -> torch.Tensor:
    """Dirichlet(1, ..., 1) rows over the last axis, fp64: normalised i.i.d. Exp(1) draws."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    e = torch.empty(shape, device=device, dtype=torch.float64).exponential_(1.0, generator=g)
    return e / e.sum(dim=-1, keepdim=True)


def normal_fill(shape, seed: int, std: float, device: str | torch.device = "cpu",
                dtype=torch.bfloat16) -> torch.Tensor:
    """N(0, std) tensor, used to fill KV pages for long-context timing runs."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(std)
    return t.to(dtype)
