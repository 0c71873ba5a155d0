"""The bench's multi-process path on the CPU: world size 2 over gloo (127.0.0.1), the
barrier and the maximum over ranks that the timed region uses, and the reference arm's
non-zero ranks leaving without work."""
from __future__ import annotations

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


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier(dist)
        # rank r times 1 + 2r ms: every rank must see the slowest
        out[rank] = bench.rank_max(dist, 1.0 + 2.0 * rank)
        bench.rank_barrier(dist)
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    assert dict(out) == {0: 3.0, 1: 3.0}


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.rank_max(None, 2.5) == 2.5
    bench.rank_barrier(None)   # no process group: returns


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
