"""The multi-GPU leg of bench.py is independent replicas (the path does not
shard); its only cross-rank steps are a barrier and the max-reduction of the
timed duration.  Checked here with two gloo ranks on CPU."""

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


def _rank(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        assert bench._dist() == (ws, rank, rank)
        dist.barrier()
        slowest = bench.reduce_max(1.5 + rank, "cpu", ws)   # rank 1 took 2.5 s
        out[rank] = (slowest, bench.job_rate(10.0, 4, ws, slowest))
    finally:
        dist.destroy_process_group()


def test_replica_timing_takes_the_slowest_rank():
    ws = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(ws, _free_port(), out), nprocs=ws, start_method="spawn")
    assert out[0] == out[1] == (2.5, 10.0 * 4 * 2 / 2.5)


def test_single_process_needs_no_group():
    assert bench.reduce_max(3.0, "cpu", 1) == 3.0
    assert bench.job_rate(6.0, 2, 1, 3.0) == 4.0
