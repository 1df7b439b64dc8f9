"""The multi-replica timing of bench.py on two CPU ranks (gloo): every rank reports the
slowest rank's step time, and the whole-job throughput counts every rank's bytes."""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, value = bench.aggregate_over_ranks(2.0 + rank, world, 1e9, dist, torch.device("cpu"))
    results[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_bytes():
    world = 2
    mgr = mp.Manager()
    results = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
    for rank in range(world):
        ms, value = results[rank]
        assert ms == 3.0  # the slower rank's 3 ms
        assert abs(value - world * 1e9 / 3e-3 / 1e9) < 1e-9  # 2 GB over 3 ms


def test_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.aggregate_over_ranks(4.0, 1, 2e9, None, None) == (4.0, 2e9 / 4e-3 / 1e9)
