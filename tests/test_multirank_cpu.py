"""The N-GPU bench path without GPUs: two gloo ranks on the CPU.

The verify round runs as independent replicas (no exchange step at B*W rows per
GPU), so the multi-GPU logic is the whole-job aggregation -- the slowest rank's
time and the sum of all ranks' tokens -- and the reference arm's rule that only
rank 0 runs and prints."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: 10 + r ms for 100 * (r + 1) tokens
        ms, tokens = bench.whole_job(10.0 + rank, 100.0 * (rank + 1))
        results[rank] = (ms, tokens)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_whole_job_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as manager:
        results = manager.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True,
                           start_method="spawn")
        got = dict(results)
    # every rank sees the slowest rank's time and all ranks' tokens
    assert got == {0: (11.0, 300.0), 1: (11.0, 300.0)}


def test_whole_job_single_rank_is_identity():
    import bench
    assert not (dist.is_available() and dist.is_initialized())
    assert bench.whole_job(2.5, 7.0) == (2.5, 7.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(None) is None     # returns before touching its arguments
    assert buf.getvalue() == ""
