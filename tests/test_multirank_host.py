"""World-size-2 checks of the benchmark's multi-rank host logic on CPU (gloo):
the job time is the slowest rank's, and throughput is the weak-scaling sum.
No GPU and no data-path collective are involved: the quantization path shards
by whole tensors, so ranks only agree on timing."""
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank                     # rank 1 is the slow one
        got = bench.max_over_ranks(mine, dist, torch.device("cpu"))
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_max_over_ranks_gloo_world2():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1] == 15.0


def test_single_rank_passthrough_and_throughput():
    assert bench.max_over_ranks(3.5, None, None) == 3.5
    # 2 ranks x 1 GB per step x 10 steps in 1 s of the slowest rank -> 20 GB/s
    assert bench.job_throughput(2, 1e9, 10, 1000.0) == pytest.approx(20.0)
    assert bench.job_throughput(1, 1e9, 10, 1000.0) == pytest.approx(10.0)
