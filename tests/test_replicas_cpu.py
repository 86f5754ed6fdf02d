"""The N > 1 path of bench.py on CPU: world size 2 over gloo.

The layer does not shard across GPUs, so N GPUs run N independent replicas
joined only by a barrier and a max over ranks of the timed region; the
reference arm runs on rank 0 alone. These tests run that plumbing as two
processes on the host, with no GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import io, json, os, sys, contextlib
sys.path.insert(0, {root!r})
import bench
world, rank, local = bench.dist_init()
assert (world, rank, local) == (2, int(os.environ["RANK"]), int(os.environ["LOCAL_RANK"]))
bench.barrier(world)
m = bench.max_over_ranks(1.5 + rank, world)
out = io.StringIO()
with contextlib.redirect_stdout(out):
    if rank != 0:
        class A:  # the reference arm's arguments; rank 1 must return without work or output
            layers = None; warmup = 3; steps = 5; gpus = 2
        bench.run_reference(A(), world, rank)
bench.barrier(world)
import torch.distributed as dist
dist.destroy_process_group()
print(json.dumps({{"rank": rank, "max": m, "ref_output": out.getvalue()}}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_ranks_barrier_max_and_reference_rank_gate():
    pytest.importorskip("torch")
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    results = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        results.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(r["rank"] for r in results) == [0, 1]
    assert all(r["max"] == 2.5 for r in results)  # the slowest rank's time, seen by every rank
    assert all(r["ref_output"] == "" for r in results if r["rank"] == 1)
