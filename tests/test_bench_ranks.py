"""Multi-process plumbing of bench.py on the CPU (gloo, world size 2).

Under torchrun every rank runs its own replica of the layer path.  The step time
is the slowest rank's (a MAX all-reduce), and only rank 0 prints the JSON line.
The reference arm runs on rank 0 alone; the other ranks return at once."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank = dist.get_rank()
ms = [3.25, 1.5][rank]
out = {{"rank": rank, "max": bench.max_over_ranks(ms, "cpu"), "env": list(bench.dist_env())}}
dist.destroy_process_group()
print(json.dumps(out))
"""


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_is_the_slowest_replica_gloo():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        so, se = p.communicate(timeout=120)
        assert p.returncode == 0, se
        outs.append(json.loads(so.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    assert all(o["max"] == 3.25 for o in outs)
    assert sorted(tuple(o["env"]) for o in outs) == [(2, 0, 0), (2, 1, 1)]


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, "cpu") == 7.5


def test_reference_arm_returns_at_once_on_other_ranks(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        gpus, steps, warmup = 2, 1, 3

    assert bench.run_reference(Args()) == 0
    assert capsys.readouterr().out == ""
