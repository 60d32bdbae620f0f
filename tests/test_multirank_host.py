"""The multi-rank (torchrun) host logic of bench.py on CPU with the gloo
backend, world size 2: every rank runs its own replica of the workload, the
job's time is the slowest rank's and its work the sum over ranks; the
reference arm does its work on rank 0 only."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, rank_ms, units, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms, value = bench.reduce_over_ranks(rank_ms[rank], units, world, torch.device("cpu"))
        out[rank] = (ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_reduce_over_ranks_gloo_world_2():
    world, port = 2, _free_port()
    rank_ms = [2.0, 3.0]  # rank 1 is the slower replica
    units = 32768.0       # tokens per replica step
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, rank_ms, units, out), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        ms, value = out[r]
        assert ms == pytest.approx(3.0)                      # max over ranks
        assert value == pytest.approx(units * world / 3e-3)  # whole-job throughput


def test_single_rank_needs_no_process_group():
    import bench
    ms, value = bench.reduce_over_ranks(2.5, 100.0, 1, torch.device("cpu"))
    assert ms == 2.5 and value == pytest.approx(100.0 / 2.5e-3)


def test_reference_arm_works_on_rank_0_only(capsys):
    import argparse
    import bench
    args = argparse.Namespace(steps=1, warmup=0, gpus=2)
    bench.reference_arm(args, {"world": 2, "rank": 1})
    assert capsys.readouterr().out == ""
