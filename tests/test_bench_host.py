"""Host logic of bench.py's multi-process (replicas) path, on CPU: two gloo
ranks on 127.0.0.1. The routing path shards over tokens with no exchange
step, so N GPUs run N independent replicas; the only collectives are the
measurement's barrier and the maximum of the step times over ranks."""
from __future__ import annotations

import contextlib
import io
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        slowest = bench.max_over_ranks(world, 10.0 + 5.0 * rank)  # rank 1 is the slow one
        q.put((rank, slowest, bench.replica_throughput(world, 16384, slowest)))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in range(world))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    # both ranks see the maximum step time; the job's rate counts every
    # rank's tokens over that time
    assert [g[1] for g in got] == [15.0, 15.0]
    assert got[0][2] == got[1][2] == pytest.approx(2 * 16384 / 15e-3)


def test_single_rank_needs_no_collective():
    assert bench.max_over_ranks(1, 3.5) == 3.5
    bench.barrier(1)
    assert bench.replica_throughput(1, 16384, 0.08) == pytest.approx(16384 / 0.08e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    """Under torchrun every rank but 0 exits without work or output."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 3, 3

    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        assert bench.run_reference(Args()) is None
    assert out.getvalue() == ""
