"""The N > 1 host logic of bench.py on CPU (gloo, world size 2): the path has
no exchange step, so ranks are independent replicas whose timed regions are
reduced to their maximum, and the job's rate counts every rank's bytes; the
reference arm runs on rank 0 only."""

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


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        ms_max, gbs = bench.job_timing(10.0 * (rank + 1), 1e9, world, "cpu")
        out[rank] = (ms_max, gbs)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_every_rank():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        ms_max, gbs = out[r]
        assert ms_max == 20.0                       # the slower rank's timed region
        assert gbs == pytest.approx(2e9 / 0.020 / 1e9)   # both ranks' bytes over it


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_timing(4.0, 2e9, 1, "cpu") == (4.0, pytest.approx(500.0))


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    assert bench.run_reference(bench.parse()) is None
    assert capsys.readouterr().out == ""
