"""The bench's multi-rank host logic (barrier + max-over-ranks timing) on two CPU ranks with
the gloo backend.  The decode path itself shards by sequence with no exchange, so the only
collective is this timing reduction."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), PKV_DIST_BACKEND="gloo")
    import bench
    d, r, w = bench._dist()
    assert (r, w) == (rank, world)
    bench._barrier(d)
    results[rank] = bench._max_over_ranks(d, 1.5 + rank * 2.0, torch.device("cpu"))
    d.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert dict(results) == {0: 3.5, 1: 3.5}


def test_single_rank_needs_no_process_group():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    d, r, w = bench._dist()
    assert d is None and (r, w) == (0, 1)
    assert bench._max_over_ranks(None, 2.0, torch.device("cpu")) == 2.0
