"""Replica (weak-scaling) host logic of bench.py on two gloo ranks (CPU).

Each rank times its own independent replica; the job's time is the slowest
rank's and the job's throughput counts the units of every rank.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    my_ms = 10.0 + 5.0 * rank  # rank 1 is slower
    m = bench.max_over_ranks(my_ms, torch.device("cpu"))
    rate = bench.whole_job_rate(world, 4, 1e12, m, 1e12)
    out[rank] = (m, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_rate_two_ranks():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1]
    m, rate = out[0]
    assert m == 15.0
    # 2 ranks x 4 steps x 1 TFLOP in 15 ms
    assert rate == pytest.approx(2 * 4 * 1.0 / 15e-3)


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
