"""The bench's multi-GPU path is replicas only (no data exchange): each rank
runs the whole layer on its own tokens and the job throughput is all ranks'
tokens over the slowest rank's time.  Checked here with two gloo ranks on
the CPU (the aggregation is host logic)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = [3.0, 5.0][rank]
    ms, tps = bench.job_throughput(ms_local, 8192, world, device="cpu")
    out[rank] = (ms, tps)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn",
                       join=True)
    for r in range(world):
        ms, tps = out[r]
        assert ms == 5.0
        assert tps == pytest.approx(2 * 8192 / 5e-3)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.job_throughput(4.0, 1000, 1) == (4.0, 1000 / 4e-3)
