"""The multi-rank host logic of bench.py on CPU with gloo, world size 2: each rank runs
its own replica, and only the timing barrier and the max / sum reductions cross ranks."""

import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    cpu = torch.device("cpu")
    ms = 10.0 + rank  # rank 1 is the slowest
    results[rank] = (bench.max_over_ranks(ms, w, cpu), bench.sum_over_ranks(100.0 * (rank + 1), w, cpu))
    torch.distributed.destroy_process_group()


def test_two_rank_reductions():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    results = mgr.dict()
    mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
    assert results[0] == results[1] == (11.0, 300.0)
