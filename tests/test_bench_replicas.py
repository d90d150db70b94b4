"""The multi-rank bookkeeping of bench.py, run as two gloo ranks on the CPU.

Each rank of ``bench.py --gpus N`` runs an independent replica; the value is
the edges of all ranks over the slowest rank's time, and only rank 0 runs the
reference arm.  These tests drive the same helpers with world size 2.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist = bench.init_group(world)
    try:
        bench.barrier(dist)
        value, total = bench.replica_throughput(dist, world, 1000, 10, local_ms[rank])
        q.put((rank, value, total))
    finally:
        dist.destroy_process_group()


def test_replica_throughput_two_ranks():
    world, port = 2, _free_port()
    local_ms = [40.0, 125.0]                      # rank 1 is the slow one
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, local_ms, q))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, value, total in got:
        assert total == pytest.approx(125.0)      # max over ranks on every rank
        assert value == pytest.approx(2 * 1000 * 10 / 0.125)


def test_replica_throughput_single_rank():
    value, total = bench.replica_throughput(None, 1, 500, 4, 20.0)
    assert total == 20.0
    assert value == pytest.approx(500 * 4 / 0.02)


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""
