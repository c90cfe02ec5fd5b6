"""CPU oracle for the speculative-decoding verify round.  TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the verify round computes,
written in numpy float64 (acceptance decisions in float32, the precision the GPU
kernel takes them in, so that integer outcomes are comparable bit for bit).

Only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s CPU-baseline leg may
import this package.  The CUDA library never imports, links or calls it, and it
never imports the CUDA library: the two share nothing but the seeded input
generators in `speculative_decoding_verify_step_gb300.synth`.

Modules
-------
decoder  Llama-style decoder forward over a paged KV cache, the pending-token
         invariant, page allocation and commit / rollback.
accept   Greedy longest-prefix acceptance, chain rejection sampling with the
         residual resample and bonus token, the integer inverse-CDF draw, and the
         greedy token-tree walk.
metrics  Strict accept rate, accept length, the expected-tokens-per-round and
         compute-factor closed forms, tree node counts.

Parity status: every function is pinned by tests in `tests/test_oracle_*.py`
against the pages' worked examples, closed forms, exact enumeration or brute
force, except the decoder forward's arithmetic, which the pages never print:
it is pinned by mathematical identities and hand-computed component values
(see tests/test_oracle_decoder.py), not by numbers from the pages.
"""

from . import accept, decoder, metrics  # noqa: F401
