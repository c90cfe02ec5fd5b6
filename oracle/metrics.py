"""Round-level metrics and closed forms (oracle; test infrastructure only).

* Strict accept rate and accept length: "投机解码的性能收支" (speculative-decoding
  performance accounting), section 二 -- strict rate = correct drafts / proposed
  drafts with no bonus; accept length = committed tokens / verify steps,
  bonus included.
* Acceptance-rate proxy = accept length / verify width (same page, section 二;
  a CI proxy, reported under that name only).
* Expected tokens per round (1 - a^(g+1)) / (1 - a), speed-up / (g c + 1),
  compute factor (g c^ + g + 1) / E: Lecture 6 "Optimizing Autoregressive Decode",
  sections 8.1, 8.2, 8.4 and their exercise answers.
* Verify-vs-decode speed-up at gamma = 1: (1 + p) T_decode / (T_verify + T_draft)
  and its break-even: "speculative decoding verify cost", section 2.
* Tree node count for a per-level branching list: Lecture 6 section 10.3 and
  its tree exercise.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Sequence


@dataclass
class Counters:
    """Counters of the accounting page: verify steps, proposed and correct drafts,
    committed (completion) tokens."""

    verify_steps: int = 0
    proposed: int = 0
    correct: int = 0
    committed: int = 0
    history: list = field(default_factory=list)

    def record_round(self, gamma: int, accepted: Sequence[int]):
        for n in accepted:
            self.verify_steps += 1
            self.proposed += gamma
            self.correct += int(n)
            self.committed += int(n) + 1
            self.history.append(int(n))

    @property
    def strict_accept_rate(self) -> float:
        return self.correct / self.proposed if self.proposed else 0.0

    @property
    def accept_length(self) -> float:
        return self.committed / self.verify_steps if self.verify_steps else 0.0

    def width_proxy(self, width: int) -> float:
        """Accept length / verify width (a CI proxy, not an acceptance rate)."""
        return self.accept_length / width


def expected_tokens_per_round(alpha: float, gamma: int) -> float:
    """E[tokens per round] = (1 - alpha^(gamma+1)) / (1 - alpha) for i.i.d. acceptance."""
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def walltime_speedup(alpha: float, gamma: int, c: float) -> float:
    """E[tokens per round] / (gamma c + 1): verify assumed as fast as one decode step."""
    return expected_tokens_per_round(alpha, gamma) / (gamma * c + 1.0)


def compute_factor(alpha: float, gamma: int, c_hat: float = 0.0) -> float:
    """Total-arithmetic factor (gamma c^ + gamma + 1) / E[tokens per round]."""
    return (gamma * c_hat + gamma + 1.0) / expected_tokens_per_round(alpha, gamma)


def speedup_gamma1(p: float, t_decode: float, t_verify: float, t_draft: float) -> float:
    """(1 + p) T_decode / (T_verify + T_draft) for one guess per round."""
    return (1.0 + p) * t_decode / (t_verify + t_draft)


def breakeven_verify(p: float, t_decode: float, t_draft: float) -> float:
    """Largest T_verify with speculation no slower than decoding: (1 + p) T_decode - T_draft."""
    return (1.0 + p) * t_decode - t_draft


def tree_nodes(branching: Sequence[int]) -> int:
    """Draft tokens in a tree whose level-d nodes each have branching[d] children."""
    total, width = 0, 1
    for k in branching:
        width *= k
        total += width
    return total


def tree_expected_accepts(topk_hit: Sequence[float]) -> float:
    """Expected accepted drafts of a greedy tree with independent levels, where
    topk_hit[d] is the probability that the right token is among the children at
    depth d+1: sum over d of prod_{e<=d} topk_hit[e]."""
    total, prod = 0.0, 1.0
    for h in topk_hit:
        prod *= h
        total += prod
    return total
