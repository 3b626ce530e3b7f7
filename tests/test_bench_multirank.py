"""The benchmark's multi-rank aggregation (replicas, max over ranks of the time,
sum of the work) with world_size 2 on CPU (gloo)."""
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


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        secs = [0.5, 0.75][rank]
        done = [1000.0, 3000.0][rank]
        results[rank] = bench.job_totals(secs, done, world, torch.device("cpu"))
    finally:
        dist.destroy_process_group()


def test_two_rank_totals_take_max_time_and_sum_work():
    mgr = mp.Manager()
    results = mgr.dict()
    port = _free_port()
    mp.spawn(_worker, args=(2, port, results), nprocs=2, join=True)
    assert results[0] == (0.75, 4000.0)
    assert results[1] == (0.75, 4000.0)


def test_single_rank_totals_are_identity():
    assert bench.job_totals(0.25, 123.0, 1, torch.device("cpu")) == (0.25, 123.0)
