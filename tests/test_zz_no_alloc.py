"""The allocation-free greedy acceptance entry point (spec_accept_greedy_noalloc).

It exists for callers that cannot call cudaMalloc: code that runs inside another
framework's memory pool or under a fixed memory budget, or a server that must not
allocate once it is serving.  Its scratch is a fixed array inside the library's
device memory.  This test calls it through the C ABI twice in a row, on different
inputs, and checks it returns exactly what spec_accept_greedy returns; it also
checks the size limit is refused on the host.  It sits in its own file, collected
last, and passes both alone in a fresh process and after the other tests."""
import numpy as np
import pytest
import torch

from tests._gpu import need_gpu

pytestmark = pytest.mark.gpu


def _case(B, gamma, V, seed):
    rng = np.random.default_rng(seed)
    logits = rng.normal(size=(B, gamma + 1, V)).astype(np.float32)
    logits[:, :, 3] = logits.max(-1) + 0.5            # ties at the top on every other row
    logits[::2, :, 11] = logits[::2, :, 3]
    am = logits.argmax(-1)
    x = np.where(rng.random((B, gamma)) < 0.6, am[:, :gamma], rng.integers(0, V, (B, gamma)))
    return torch.from_numpy(logits).cuda(), torch.from_numpy(x).cuda()


def test_noalloc_matches_greedy_accept_twice_in_a_row():
    need_gpu()
    from speculative_decoding_verify_step_gb300 import spec
    dev = torch.device("cuda")
    for B, gamma, V, seed in [(64, 7, 128256, 1), (255, 15, 1024, 2)]:
        logits, x = _case(B, gamma, V, seed)
        want = spec.spec_accept_greedy(logits, x)
        outs = tuple(torch.full_like(t, -7) for t in want)
        got = spec.spec_accept_greedy_noalloc(logits, x, outs=outs)
        for g, w in zip(got, want):
            assert torch.equal(g, w)
    assert dev.type == "cuda"


def test_noalloc_refuses_more_rows_than_its_scratch():
    need_gpu()
    from speculative_decoding_verify_step_gb300 import spec
    logits = torch.zeros(257, 16, 128, device="cuda")     # 4112 rows > 4096
    with pytest.raises(spec.SpecError) as e:
        spec.spec_accept_greedy_noalloc(logits, torch.zeros(257, 15, dtype=torch.int32, device="cuda"))
    assert e.value.status == 1
