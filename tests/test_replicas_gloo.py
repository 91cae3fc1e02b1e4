"""Multi-process (replicas) aggregation of bench.py on CPU: two gloo ranks.

The GEMM does not shard across GPUs here (one GPU per process, independent
replicas); what crosses ranks is the timing reduction: each shape's time is
the max over ranks and the whole-job value counts every rank's work.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, sizes, per_rank_times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        times, value = bench.replica_value(sizes, per_rank_times[rank], world, "cpu")
        out[rank] = (times, value)
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_max_time_and_count_both():
    sizes = [1024, 2048, 4096]
    per_rank = [[0.020, 0.050, 0.120], [0.025, 0.040, 0.130]]
    world = 2
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_worker, args=(world, _free_port(), sizes, per_rank, out), nprocs=world,
                 join=True)
        res = dict(out)
    worst = [max(a, b) for a, b in zip(*per_rank)]
    want = bench.geomean([world * 2.0 * s ** 3 / t / 1e9 for s, t in zip(sizes, worst)])
    for rank in range(world):
        times, value = res[rank]
        assert times == pytest.approx(worst)
        assert value == pytest.approx(want)


def test_single_replica_needs_no_process_group():
    times, value = bench.replica_value([2048], [0.05], 1, "cpu")
    assert times == [0.05]
    assert value == pytest.approx(2.0 * 2048 ** 3 / 0.05 / 1e9)
