"""Host-side logic of the multi-rank benchmark path, on CPU with gloo (world size 2):
each rank draws an independent batch of heads, and the job's time is the
maximum over ranks."""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    w = wl.Workload("mr", 1, 64, 2, 64, "bf16", 7, gate="normal", lo=1.0, backward=True)
    arrays = bench.draw_inputs(w, rank)
    slowest = bench.max_over_ranks(1.5 + rank, dist)
    out[rank] = (float(arrays["q"].astype(np.float64).sum()), slowest)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_draw_distinct_batches_and_take_max_time():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][1] == res[1][1] == 2.5
    assert res[0][0] != res[1][0]


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks(3.25) == 3.25
