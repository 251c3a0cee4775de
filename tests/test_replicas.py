"""The multi-GPU path of bench.py runs one replica of the step per rank and
needs no data-path collective: only the per-step time is reduced (MAX over
ranks) and the job rate counts every rank's work.  Checked here with two gloo
ranks on the CPU, plus the reference arm's rule that only rank 0 runs it."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 1.0 + 2.0 * rank  # rank 1 is the slow replica
        slowest = bench.max_over_ranks(local_ms)
        out[rank] = (slowest, bench.job_tflops(1e12, world, slowest))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_replica():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    for rank in range(world):
        slowest, tflops = out[rank]
        assert slowest == pytest.approx(3.0)
        # 1e12 FLOP per rank and step, two ranks, 3 ms: 2e12 / 3e-3 / 1e12 TFLOP/s
        assert tflops == pytest.approx(2e12 / 3e-3 / 1e12)


def test_single_process_uses_its_own_time():
    import bench

    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.job_tflops(1e12, 1, 2.0) == pytest.approx(500.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import argparse

    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(workload=1, ref_rows=8, steps=1, warmup=0)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
