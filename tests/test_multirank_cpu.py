"""The multi-GPU path of bench.py is one pool replica per rank (weak scaling)
with no data-path collective; the only cross-rank step is the max of the
timings.  Checked here with two gloo ranks on CPU."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 10.0 - rank, 0.5 * (rank + 1)]
        out[rank] = bench.max_over_ranks(mine, dist, torch.device("cpu"))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        got = dict(out)
    for r in range(world):
        assert got[r] == [2.0, 10.0, 1.0]
