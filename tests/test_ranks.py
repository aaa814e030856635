"""The multi-process path of the benchmark on CPU: two gloo ranks reduce their
per-rank times to the maximum, and the whole-job throughput counts every
rank's replica (the GEMM itself shards as independent replicas, with no
collective on the data path)."""
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


def _worker(rank, world, port, queue):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [1.0 + rank, 10.0 - rank, 5.0]
        queue.put((rank, bench.reduce_job_times(local, world, "cpu")))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_maximum_time():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0] == results[1] == [2.0, 10.0, 5.0]


def test_job_tflops_counts_every_replica():
    # 1 TFLOP per step, 10 steps, 2 ranks, 1 s -> 20 TFLOP/s
    assert bench.job_tflops(1e12, 10, 2, 1000.0) == pytest.approx(20.0)
    assert bench.job_tflops(1e12, 10, 1, 1000.0) == pytest.approx(10.0)


def test_single_rank_needs_no_process_group():
    assert bench.reduce_job_times([3.0, 4.0], 1, "cpu") == [3.0, 4.0]
