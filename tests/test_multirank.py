"""The N > 1 host path of bench.py on CPU: two gloo ranks with different timings agree on
the max over ranks, and the reference arm does its work on rank 0 only."""
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


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        mine = [1.0 + rank, 5.0 - rank, 2.0 * (rank + 1)]
        res = bench.max_over_ranks(mine, device="cpu")
        out[rank] = res
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == [2.0, 5.0, 4.0]
    assert out[1] == [2.0, 5.0, 4.0]


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 1.5]) == [3.0, 1.5]


def test_reference_arm_runs_on_rank0_only(capsys):
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    args = argparse.Namespace(gpus=2, steps=1, warmup=0)
    bench.run_reference(args, rank=1, world=2)      # not rank 0: returns without work
    assert capsys.readouterr().out == ""
