"""The multi-GPU path of the benchmark on the CPU: world size 2 over gloo.

Requests shard across GPUs with no data exchange (each rank runs its own
replica), so the only cross-rank steps are the barrier, the max of the ranks'
timed seconds and the sum of their injected bytes.  These run here on CPU
ranks; nothing touches a GPU.
"""
import os
import socket

import pytest
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
    os.environ["RANK"] = str(rank)
    os.environ["WORLD_SIZE"] = str(world)
    os.environ["LOCAL_RANK"] = str(rank)
    r, w, local = bench.dist_env()
    d = bench.dist_init(w, "gloo")
    assert d is not None and d.get_world_size() == world and r == rank
    bench.barrier(d)
    my_time = 1.0 + rank            # rank 1 is the slow one
    my_bytes = 100.0 * (rank + 1)
    t = bench.max_over_ranks(d, my_time)
    b = bench.sum_over_ranks(d, my_bytes)
    out[rank] = (t, b, bench.replica_seed(1, rank))
    d.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as man:
        out = man.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.0          # max of the ranks' times
    assert res[0][1] == res[1][1] == 300.0        # bytes of all ranks
    assert res[0][2] != res[1][2]                 # independent replicas


def test_single_rank_needs_no_process_group():
    assert bench.dist_init(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.sum_over_ranks(None, 7.0) == 7.0
