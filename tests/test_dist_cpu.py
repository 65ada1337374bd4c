"""bench.py's multi-rank host logic on CPU: two gloo ranks, barrier and the
max-over-ranks reduction of the step time.  Every rank runs its own copy of
the workload (independent chains), so this reduction is the only exchange."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist
    import bench
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        bench.barrier(world)
        got = bench.reduce_max(1.5 + 2.0 * rank, world)
        results[rank] = got
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        assert dict(results) == {0: 3.5, 1: 3.5}


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(2.25, 1) == 2.25
