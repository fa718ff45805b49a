"""The benchmark's multi-GPU logic on CPU processes (gloo, world size 2):
the job time is the slowest rank's (max over ranks), every rank runs its
own sequence of decode steps (replicas; the method is single-GPU), and one
process alone reduces to the identity."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        mine = [10.0 + rank, 5.0 - rank]  # rank 1 slower on the first, faster on the second
        got = bench.reduce_max_over_ranks(mine, world, device="cpu")
        q.put((rank, got, bench.replica_steps(rank, 8, 256)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_distinct_replica_steps():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict()
    for _ in range(2):
        r, got, steps = q.get(timeout=120)
        res[r] = (got, steps)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == res[1][0] == [11.0, 5.0]
    assert res[0][1] != res[1][1] and len(set(res[0][1])) == 8


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
