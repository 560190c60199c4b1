"""Multi-process paths of bench.py on CPU (gloo, world size 2).

The layer does not shard: several GPUs run independent replicas, and the only
cross-rank steps are the barrier around the timed region and the max over
ranks of the step time.  These tests run those steps, and the reference arm
under torch.distributed.run, as two CPU processes.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ranks_agree(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # rank r reports a step time of 1 + r ms: every rank must see the slowest
        q.put((rank, bench.max_over_ranks(1.0 + rank, world, torch.device("cpu"))))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_processes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ranks_agree, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 2.0, 1: 2.0}


def test_reference_arm_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "small_T8",
           "--gpus", "2", "--steps", "3", "--warmup", "3", "--ref-budget-s", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout   # rank 0 alone prints
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2
    assert res["value"] > 0 and res["e2e"]["h2d_bytes_per_step"] == 0
    assert res["cpu_baseline"]["kind"] == "oracle"
