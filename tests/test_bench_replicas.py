"""The N > 1 path of bench.py on CPU: two gloo ranks, each a replica with its
own time; the job's throughput uses the slowest rank."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = 1.0 + rank          # rank 1 is the slow replica
        tmax = bench.max_over_ranks(t, dist)
        v = bench.replica_throughput(2e12, 3, world, tmax)
        q.put((rank, tmax, v))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_use_max_time_and_sum_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, tmax, v in res:
        assert tmax == 2.0                       # the slower rank's time
        assert abs(v - 2 * 2e12 * 3 / 2.0 / 1e12) < 1e-12


def test_single_process_is_identity():
    assert bench.max_over_ranks(1.5, None) == 1.5
    assert bench.replica_throughput(1e12, 2, 1, 2.0) == 1.0
