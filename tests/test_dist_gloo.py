"""The bench's multi-rank host logic (barrier + max-over-ranks timing, and the launcher that
`--gpus N` starts) on two CPU ranks with the gloo backend.  The decode path itself shards by
sequence with no exchange, so the only collective is this timing reduction."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

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


def _bench_env(**extra):
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env.update(PKV_DIST_BACKEND="gloo", **extra)
    return env


def test_bench_gpus_n_launches_n_ranks():
    """`bench.py --gpus 2` run directly starts two ranks itself (torch.distributed.run on
    127.0.0.1); they meet at the barrier and rank 0 reports both ranks and the max over ranks."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--dist-check"],
                       capture_output=True, text=True, timeout=300, env=_bench_env(), cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert lines == [{"dist_check": {"world": 2, "ranks": [0, 1], "max_over_ranks": 2.0}}]


def test_bench_refuses_a_world_size_other_than_gpus():
    """A rank started with WORLD_SIZE different from --gpus exits non-zero instead of timing and
    printing a line whose n_gpus disagrees with the request."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--dist-check"],
                       capture_output=True, text=True, timeout=120, cwd=ROOT,
                       env=_bench_env(WORLD_SIZE="1", RANK="0", LOCAL_RANK="0"))
    assert r.returncode != 0
    assert "WORLD_SIZE=1" in r.stderr
