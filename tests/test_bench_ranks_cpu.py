"""bench.py's multi-rank host logic on CPU ranks (gloo, world size 2).

Each rank runs its own copy of the workload (replicas, no data-path collective); the job's
throughput is every rank's work over the slowest rank's time, and only rank 0 prints.
"""

from __future__ import annotations

import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench.dist_info()
        reduce_max, barrier = bench.make_collectives(w, "cpu")
        barrier()
        # rank r "took" 1 + r seconds for 10 units of work
        value, t_max = bench.aggregate(1.0 + r, 10.0, w, reduce_max)
        barrier()
        results[r] = (r, w, value, t_max)
    finally:
        dist.destroy_process_group()


def test_two_ranks_aggregate_over_the_slowest():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as manager:
        results = manager.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        got = dict(results)
    assert set(got) == {0, 1}
    for r in range(2):
        rank, world, value, t_max = got[r]
        assert (rank, world) == (r, 2)
        assert t_max == 2.0                    # the slowest rank's time, on every rank
        assert value == pytest.approx(10.0)    # 2 ranks x 10 units / 2 s


def test_single_rank_collectives_are_identity():
    reduce_max, barrier = bench.make_collectives(1, "cpu")
    assert reduce_max(3.5) == 3.5 and barrier() is None
    assert bench.aggregate(0.5, 8.0, 1, reduce_max) == (16.0, 0.5)


def test_reference_arm_other_ranks_exit_quietly(monkeypatch):
    """Under torchrun only rank 0 times the oracle and prints; rank 1 exits 0 with no output."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.run_reference(type("A", (), {"steps": 2, "warmup": 1})())
    assert rc == 0 and buf.getvalue() == ""
