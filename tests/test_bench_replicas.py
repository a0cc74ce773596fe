"""bench.py's multi-rank bookkeeping on CPU: the max-over-ranks time that
the whole-job throughput divides by, over a world of 2 gloo ranks."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out[rank] = bench.reduce_max(torch, dist, 1.5 + rank, torch.device("cpu"))
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    ctx_procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in ctx_procs:
        p.start()
    for p in ctx_procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_reduce_max_single_process_is_identity():
    import bench
    assert bench.reduce_max(torch, dist, 3.25, torch.device("cpu")) == 3.25
