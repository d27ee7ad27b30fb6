"""Multi-GPU use is replicas only: every rank runs its own requests, and the
benchmark combines ranks by taking the slowest rank's time and the sum of
all ranks' tokens.  That host logic runs here on two gloo ranks (CPU)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                            rank=rank, world_size=world)
    try:
        # rank r ran for 10 (r + 1) ms and processed 3136 (r + 1) tokens
        ms, tokens = bench.combine_ranks(10.0 * (rank + 1), 3136 * (rank + 1))
        q.put((rank, ms, tokens))
    finally:
        dist.destroy_process_group()


def test_two_replicas_combine_with_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms, tokens in got:
        assert ms == 20.0            # the slowest replica bounds the job
        assert tokens == 3 * 3136    # every replica's work counts


def test_single_process_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.combine_ranks(12.5, 3136) == (12.5, 3136)
