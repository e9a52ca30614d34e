"""The N > 1 path (replicas only): two gloo ranks on the CPU.

Each rank runs an independent replica; the job's step time is the slowest
rank's and its throughput is all ranks' tokens over that time.  The reference
arm does its work on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, value = bench.replica_throughput(10.0 + 5.0 * rank, 100, dist, torch.device("cpu"))
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_max_time_and_summed_tokens():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(world))
    for _, ms, value in out:
        assert ms == pytest.approx(15.0)  # the slower rank sets the step time
        assert value == pytest.approx(2 * 100 / 0.015)  # both ranks' tokens over it


def test_single_process_throughput():
    import bench

    ms, value = bench.replica_throughput(4.0, 32)
    assert ms == 4.0 and value == pytest.approx(8000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench

    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(None) == 0
    assert capsys.readouterr().out == ""
