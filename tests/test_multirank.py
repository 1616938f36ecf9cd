"""bench.py's multi-rank host logic on CPU: two gloo ranks rendezvous on
127.0.0.1, meet at the barrier, agree on the max over ranks, and only rank
0 of the reference arm does work (the other ranks return at once)."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import json, os, sys, time
sys.path.insert(0, sys.argv[1])
import bench
rank, world, local = bench.dist_setup()
bench.barrier(world)
m = bench.max_over_ranks(1.5 + rank, world)
t = time.perf_counter()
class A: steps = 1; warmup = 0; workload = "decode_12x3_d64_L1024"
if rank != 0:
    bench.run_reference(A())          # must return without work
ref_s = time.perf_counter() - t
bench.barrier(world)
print(json.dumps({"rank": rank, "world": world, "max": m, "ref_s": ref_s}), flush=True)
import torch.distributed as td
td.destroy_process_group()
"""


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_barrier_and_max(tmp_path):
    pytest.importorskip("torch")
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT, ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=240)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    assert all(o["world"] == 2 and o["max"] == 2.5 for o in outs)
    assert next(o for o in outs if o["rank"] == 1)["ref_s"] < 1.0
