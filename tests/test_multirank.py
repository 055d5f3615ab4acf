"""Multi-process host logic of bench.py (N > 1 replicas): rank rendezvous,
barrier and the max-over-ranks reduction of the per-step time, on gloo with
world size 2 on the CPU."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    d, r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    dev = torch.device("cpu")
    d.barrier()
    # each rank reports its own step time; every rank must see the slowest one
    t = bench.max_over_ranks(d, 1.5 + rank, dev)
    out[rank] = t
    d.destroy_process_group()


def test_two_rank_max_over_ranks():
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_process_needs_no_group():
    os.environ.pop("WORLD_SIZE", None)
    d, r, w, local = bench.dist_setup(1)
    assert d is None and (r, w) == (0, 1)
    assert bench.max_over_ranks(None, 3.0, torch.device("cpu")) == 3.0
