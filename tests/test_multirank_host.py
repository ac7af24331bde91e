"""The multi-GPU path is independent replicas (one process per GPU, no data
collective): the job's time is the slowest rank's and the value counts every
rank's work.  These tests run that host logic as world-size-2 gloo ranks on
the CPU (no GPU)."""
import os
import socket
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


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    seconds = [0.5, 2.0][rank]  # rank 1 is the slow one
    t = bench.max_over_ranks(seconds, dist)
    v = bench.job_throughput(world, 100, 3.0, t)
    dist.barrier()
    results[rank] = (t, v)
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_every_rank():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        res = dict(results)
    for rank in range(world):
        t, v = res[rank]
        assert t == 2.0  # every rank sees the slowest rank's time
        assert v == pytest.approx(world * 100 * 3.0 / 2.0)


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, None) == 1.25
    assert bench.job_throughput(1, 10, 2.0, 4.0) == 5.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun every rank but 0 exits at once without work or output."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")

    class Args:
        workload = "tiny"
        steps = 1
        warmup = 0
        gpus = 2
        ref_seconds = 0.1
    assert bench.run_reference(Args()) == 0
    assert capsys.readouterr().out == ""
