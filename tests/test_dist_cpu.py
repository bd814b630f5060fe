"""The multi-process path of bench.py on CPU (gloo, world size 2).

Decode attention shards by (sequence, KV head) with no exchange, so N GPUs
run N independent replicas: the reported time is the maximum over ranks and
the token count the sum.  These tests run those reductions, and the
reference arm under torchrun (rank 0 prints one line, the other rank exits
cleanly), as two gloo processes without a GPU."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _reduce_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [3.5, 7.25][rank]
        tokens = [100.0, 250.0][rank]
        out[rank] = (bench.max_over_ranks(elapsed, world, "cpu"), bench.sum_over_ranks(tokens, world, "cpu"))
        bench.barrier(world)
    finally:
        torch.distributed.destroy_process_group()


def test_rank_reductions_two_processes():
    """Max of the ranks' times, sum of their tokens, seen by every rank."""
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_reduce_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1] == (7.25, 350.0)


def test_reference_arm_under_torchrun_two_ranks():
    """bench.py --impl reference launched the way the multi-GPU run is:
    exactly one JSON line (from rank 0), exit status 0 on every rank."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=240)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
