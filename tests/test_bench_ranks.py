"""Host logic of multi-GPU bench runs on CPU: two gloo ranks (127.0.0.1) take the barrier and
the maximum of their per-rank times the way bench.py's replicas do, and the whole-job value
counts every replica's bytes over the slowest replica's time.  The reference arm's other ranks
exit without work."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        group = bench.RankGroup(world, torch.device("cpu"))
        group.barrier()
        ms = group.max(10.0 + 3.0 * rank)  # the slower rank decides
        group.barrier()
        out[rank] = ms
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert out[0] == out[1] == 13.0


def test_job_value_counts_all_replicas():
    sys.path.insert(0, ROOT)
    import bench
    b = 11_305_601_024
    one = bench.job_value(1, b, 2.5)
    assert one == pytest.approx(b / 2.5e-3 / 1e9)
    assert bench.job_value(4, b, 2.5) == pytest.approx(4 * one)
    assert bench.RankGroup(1, torch.device("cpu")).max(7.0) == 7.0


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"])
    bench.run_reference(bench.parse_args())
    assert capsys.readouterr().out == ""
