"""CPU: the benchmark's multi-rank path (independent replicas, max-over-ranks timing)
with two gloo ranks."""
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
    try:
        mine = [1.0 + rank, 10.0 - rank, 3.5]
        got = bench.reduce_max(mine, world, torch.device("cpu"))
        dist.barrier()
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_reduce_max_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    want = [2.0, 10.0, 3.5]
    assert res[0] == want and res[1] == want


def test_reduce_max_single_rank_is_identity():
    assert bench.reduce_max([1.5, 2.5], 1, torch.device("cpu")) == [1.5, 2.5]


def test_whole_job_rate_counts_every_replica():
    # two replicas of 1e12 FLOP each, slowest rank 0.5 s -> 4 TFLOP/s for the job
    assert bench.whole_job_rate(1e12, 2, 500.0, 1e12) == pytest.approx(4.0)
    assert bench.whole_job_rate(1e12, 1, 500.0, 1e12) == pytest.approx(2.0)
