"""The N > 1 path on CPU: world-size-2 gloo ranks.

The verify step shards by sequence with no exchange step, so N GPUs run N
independent replicas.  What must hold across ranks is the bench's timing
contract: a barrier on both sides of the timed region and the maximum time
over ranks, and rank 0 alone printing the line.
"""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    got = bench.max_over_ranks(float(rank + 1) * 1.5, w, torch.device("cpu"))
    bench.barrier(w)
    out_q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29517
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 3.0, 1: 3.0}


def test_reference_arm_under_torchrun_world2():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=29533", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--config", "tiny_chain_ctx512", "--steps", "1", "--warmup", "0",
           "--gpus", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1                      # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "steps/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
