"""Host logic of `bench.py --gpus N` (N independent replicas): whole-job
throughput sums the units of every rank and divides by the slowest rank's
time.  Checked with two gloo ranks on the CPU."""
import os
import socket

import pytest
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
        seconds = [2.0, 3.0][rank]
        units = [100.0, 50.0][rank]
        rate, slowest = bench.aggregate(seconds, units, world, dist)
        q.put((rank, rate, slowest))
    finally:
        dist.destroy_process_group()


def test_replicas_aggregate_over_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for _, rate, slowest in got:
        assert slowest == pytest.approx(3.0)
        assert rate == pytest.approx(150.0 / 3.0)


def test_single_rank_aggregate_is_plain_ratio():
    assert bench.aggregate(2.0, 10.0, 1, None) == (5.0, 2.0)


def test_algorithmic_bytes_of_the_large_workload():
    ab = bench.algorithmic_bytes(T=16384, H=7168, N=47341, K=8, P=8)
    row = 7168 * 2
    assert ab["dispatch"] == 16384 * row + 47341 * row + 16384 * 8 * 4
    assert ab["combine"] == 47341 * row + 16384 * row + 16384 * 8 * 4
