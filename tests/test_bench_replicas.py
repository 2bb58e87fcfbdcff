"""The multi-GPU form of the bench is N independent replicas (the step has no
data-parallel exchange); only the timing is combined: every rank reports the
maximum over ranks.  Checked here with two gloo processes on the CPU."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    vals = bench.max_over_ranks(dist, [1.0 + rank, 10.0 - rank])
    out[rank] = vals
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_processes():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    port = 29600 + os.getpid() % 200
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == [2.0, 10.0]
    assert out[1] == [2.0, 10.0]


def test_max_over_ranks_without_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, [3.0, 4.0]) == [3.0, 4.0]
