"""The multi-rank plumbing of bench.py on CPU (gloo, world size 2): ranks
time their own tokens, the slowest rank's time decides, the aggregate counts
every rank's tokens.  No data-path collective is involved."""
import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.dist_init(world, use_cuda=False)
    bench.barrier(world)
    my_ms = 100.0 * (rank + 1)              # rank 1 is the slow one
    slowest = bench.max_over_ranks(my_ms, world, torch.device("cpu"))
    value = bench.aggregate(tokens_per_rank=4096, steps=10, world=world, max_total_ms=slowest)
    out[rank] = (slowest, value)
    torch.distributed.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        slowest, value = out[r]
        assert slowest == 200.0
        assert abs(value - 2 * 4096 * 10 / 0.2) < 1e-6
