"""The benchmark's multi-process path (replicas, max-over-ranks timing,
whole-job aggregation) on two gloo ranks on the CPU."""
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


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_env()
        assert (w, r, lr) == (world, rank, rank)
        bench.barrier(world)
        ms = bench.reduce_max(times[rank], world, torch.device("cpu"))
        out[rank] = ms
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    times = [1.5, 2.5]
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, times, out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == max(times)
    import bench
    # 2 replicas, each 1 GB per step, slowest rank 2.5 ms per step
    assert bench.aggregate(1e9, max(times), world, "GB/s") == pytest.approx(2 * 1e9 / 2.5e-3 / 1e9)
    assert bench.aggregate(2e12, 1.0, 1, "TFLOP/s") == pytest.approx(2000.0)


def test_single_rank_needs_no_process_group(monkeypatch):
    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    assert bench.dist_env()[0] == 1
    assert bench.reduce_max(3.0, 1, torch.device("cpu")) == 3.0
    bench.barrier(1)
