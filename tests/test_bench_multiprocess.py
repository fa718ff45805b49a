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


def test_reference_arm_json_contract():
    """``bench.py --impl reference`` (the CPU oracle on a bounded sample)
    prints one JSON line with the contract's keys, on a host without a GPU."""
    import json
    import subprocess

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--cpu-layers", "1"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ["impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"]:
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] >= 3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("gptoss20b_decode")
