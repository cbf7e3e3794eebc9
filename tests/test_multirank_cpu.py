"""The multi-process parts of bench.py on CPU: two gloo ranks (one process per GPU on a
multi-GPU node; here plain processes) agree on the slowest rank's time, and the job's value is
every rank's tokens over that time. The reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench

    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, torch.device("cpu"))
        q.put((rank, ms, bench.job_throughput(world, 4096, 10, ms)))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, ms, value in got:
        assert ms == 15.0  # the slower rank's 15 ms, on both ranks
        assert value == pytest.approx(2 * 4096 * 10 / 0.015)


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(12.5, 1, torch.device("cpu")) == 12.5
    assert bench.job_throughput(1, 4096, 200, 1000.0) == pytest.approx(4096 * 200)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = bench.parse(["--impl", "reference", "--gpus", "2"])
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""  # no work, no line on the other ranks
