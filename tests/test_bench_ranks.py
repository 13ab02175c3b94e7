"""bench.py's multi-rank plumbing and its CPU reference arm, on the CPU.

Under torchrun each rank runs an independent replica and the timed region is the maximum
over ranks; this is checked with two gloo ranks.  The reference arm (the CPU oracle on a
bounded sample of the step) runs end to end here and must print one JSON line; under
torchrun only rank 0 prints.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    mine = 10.0 + 5.0 * rank  # rank 1 is the slow one
    q.put((rank, bench.reduce_max(mine, torch.device("cpu"))))
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def test_reduce_max_single_process():
    import torch
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, torch.device("cpu")) == 3.5


def _reference(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                           "--steps", "2", "--warmup", "1", *args], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=600)


def test_reference_arm_prints_one_line():
    r = _reference({})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["workload"] == "tiny"


def test_reference_arm_other_ranks_print_nothing():
    r = _reference({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def _rank_fails(rank, world, port, q):
    import datetime
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=10))
    import bench

    if rank == 1:
        os._exit(3)  # this rank dies between steps, before the timing reduction
    import time
    t0 = time.time()
    try:
        bench.reduce_max(1.0, torch.device("cpu"))
        outcome = "returned"
    except Exception as e:  # the survivor learns of the failure instead of waiting forever
        outcome = type(e).__name__
    q.put((rank, outcome, time.time() - t0))
    q.close()
    q.join_thread()  # flush the message before leaving without tearing down the broken group
    os._exit(0)


def test_a_dead_rank_fails_the_reduction_instead_of_hanging():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_fails, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert procs[1].exitcode == 3
    rank, outcome, secs = q.get(timeout=10)
    assert rank == 0 and outcome != "returned" and secs < 60, (outcome, secs)
