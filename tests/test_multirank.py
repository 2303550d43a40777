"""The bench's multi-rank timing helpers on two CPU ranks (gloo backend).

bench.py under torchrun runs one independent replica per GPU (the layer needs
no exchange on one GPU per problem); the only cross-rank steps are the
barrier around the timed region and the max over ranks of the step time.
These run here as two spawned processes on the gloo backend.
"""
from __future__ import annotations

import os
import socket

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, queue) -> None:
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(world)
        slowest = bench.max_over_ranks(world, 0.5 + rank)  # rank 1 is the slow one
        bench.barrier(world)
        queue.put((rank, slowest))
    finally:
        dist.destroy_process_group()


def test_barrier_and_max_over_ranks_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = dict(queue.get(timeout=5) for _ in procs)
    assert got == {0: 1.5, 1: 1.5}


def test_single_rank_helpers_are_identities():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    bench.barrier(1)
    assert bench.max_over_ranks(1, 2.25) == 2.25
