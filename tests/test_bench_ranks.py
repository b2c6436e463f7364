"""The bench's multi-process aggregation (replicas only), on CPU with gloo, world size 2."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 100.0 + 50.0 * rank  # rank 1 is the slow one
    m = bench.max_over_ranks(ms, dist, torch.device("cpu"))
    v = bench.whole_job_tflops(world, 2e12, 4, m)
    out[rank] = (m, v)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 150.0
    # 2 replicas x 4 steps x 2e12 FLOPs over 150 ms
    assert out[0][1] == pytest.approx(2 * 4 * 2e12 / 0.150 / 1e12)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.whole_job_tflops(1, 1e12, 1, 1000.0) == pytest.approx(1.0)
