"""The bench's whole-job reduction over ranks, run as two gloo ranks on the
CPU: the time is the slowest rank's, the bytes are summed."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, nb = bench.reduce_over_ranks(dist, 10.0 + 5.0 * rank, 1000 * (rank + 1))
        out[rank] = torch.tensor([ms, nb], dtype=torch.float64)
    finally:
        dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    world = 2
    out = torch.zeros((world, 2), dtype=torch.float64).share_memory_()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    for r in range(world):
        assert out[r, 0].item() == 15.0          # max over ranks
        assert out[r, 1].item() == 3000.0        # sum over ranks


def test_reduce_single_rank():
    assert bench.reduce_over_ranks(None, 7.5, 42) == (7.5, 42.0)
