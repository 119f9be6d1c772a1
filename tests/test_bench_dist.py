"""The benchmark's multi-rank host logic with world size 2 on CPU (gloo).

Each rank runs its own micro-batch; the job's throughput is every rank's
FLOPs over the slowest rank's time, and the ranks only exchange the timing
numbers (no collective on the data path).
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


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [0.50, 0.75][rank]
    flops = [3.6e11, 4.5e11][rank]
    ms_max, total = bench.aggregate(dist, torch, ms, flops, torch.device("cpu"))
    results[rank] = (ms_max, total, bench.whole_job_tflops(total, ms_max))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    for rank in range(world):
        ms_max, total, value = res[rank]
        assert ms_max == pytest.approx(0.75)
        assert total == pytest.approx(8.1e11)
        assert value == pytest.approx(8.1e11 / 0.75e-3 / 1e12)


def test_dist_setup_reads_torchrun_env(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "4")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.dist_setup(None) == (1, 4, 1)
