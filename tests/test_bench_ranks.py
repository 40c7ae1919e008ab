"""Multi-rank logic of bench.py, run as two gloo ranks on the CPU: the step time is the slowest rank's,
the rate counts every rank's work, and the reference arm prints on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 20.0][rank]                      # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, dist, "cpu")
        rate = bench.whole_job_rate(1.0e9, world, ms)
        out[rank] = (ms, rate)
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_step_time_two_gloo_ranks():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()          # no fork of this multi-threaded process
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    for rank in range(world):
        ms, rate = out[rank]
        assert ms == 20.0
        assert rate == pytest.approx(2 * 1.0e9 / 0.020)


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_rate(5.0, 1, 1000.0) == pytest.approx(5.0)


def test_reference_arm_is_silent_on_other_ranks(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(argparse.Namespace(steps=1, warmup=0))
    assert capsys.readouterr().out == ""
