"""Multi-process host logic of bench.py (N > 1, a batch per rank): rank
rendezvous, barrier, the max-over-ranks reduction of the per-step time and the
sum of the ranks' work, on gloo with world size 2 on the CPU."""
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
    # and the job's work is the sum of every rank's own batch
    f = bench.sum_over_ranks(d, 10.0 * (rank + 1), dev)
    out[rank] = (t, f)
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
    assert dict(out) == {0: (2.5, 30.0), 1: (2.5, 30.0)}


def test_single_process_needs_no_group():
    os.environ.pop("WORLD_SIZE", None)
    d, r, w, local = bench.dist_setup(1)
    assert d is None and (r, w) == (0, 1)
    assert bench.max_over_ranks(None, 3.0, torch.device("cpu")) == 3.0
    assert bench.sum_over_ranks(None, 3.0, torch.device("cpu")) == 3.0


def test_rank_batches_differ_rank0_keeps_the_workload():
    """Each rank draws its own batch of the workload's shape; rank 0's is the
    workload itself."""
    from ragged_varlen_attention_gb300 import workloads as wl
    base = wl.WORKLOAD_SEEDS["padded_causal"]
    assert bench.rank_seed(base, 0) == base
    b0 = wl.make("padded_causal", seed=bench.rank_seed(base, 0), b=3, h=2, max_len=200)
    ref = wl.make("padded_causal", b=3, h=2, max_len=200)
    b1 = wl.make("padded_causal", seed=bench.rank_seed(base, 1), b=3, h=2, max_len=200)
    assert torch.equal(b0.q.view(torch.uint8), ref.q.view(torch.uint8))
    assert b1.q.shape != ref.q.shape or not torch.equal(b1.q.view(torch.uint8), ref.q.view(torch.uint8))
