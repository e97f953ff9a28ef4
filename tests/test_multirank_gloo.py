"""The benchmark's N > 1 host logic on two gloo ranks (CPU): every rank runs its
own replica, rank 0 reports the bytes of all ranks over the slowest rank's
time.  No GPU and no data-path collective are involved."""
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


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r moved (r + 1) GB in (r + 1) * 0.5 s
    gbps, t_max, n = bench.aggregate_over_ranks((rank + 1) * 1e9, (rank + 1) * 0.5, dist, "cpu")
    out[rank] = torch.tensor([gbps, t_max, n], dtype=torch.float64)
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_two_ranks():
    world = 2
    out = torch.zeros(world, 3, dtype=torch.float64).share_memory_()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    # total 3 GB over the slowest rank's 1.0 s = 3 GB/s, same answer on both ranks
    for r in range(world):
        assert out[r, 0].item() == pytest.approx(3.0)
        assert out[r, 1].item() == pytest.approx(1.0)
        assert out[r, 2].item() == 2


def test_aggregate_single_process():
    import bench
    gbps, t_max, n = bench.aggregate_over_ranks(2e9, 0.5)
    assert (gbps, t_max, n) == (4.0, 0.5, 1)
