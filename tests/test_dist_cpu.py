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


def test_cpu_baseline_sample_legs():
    """The oracle legs timed beside the long-context and varlen workloads: a
    bounded prefix of sequence 0 over every head, from its initial state, on
    host cores (small shapes here, so the leg runs in well under a second)."""
    import torch
    import bench
    from hybrid_linear_attention_chunk_gb300 import inputs
    for base in (inputs.LONG_T1M, inputs.VARLEN_64):
        kw = dict(H=2, dk=16, dv=16, qkv_dtype=torch.float32, out_dtype=torch.float32)
        w = inputs.scaled(base, T=512, **kw) if base.varlen_seqs == 0 else inputs.scaled(base, varlen_seqs=3, **kw)
        x = inputs.make_prefill(w, device="cpu")
        r = bench.cpu_baseline_sample(w, x, seconds=0.2)
        assert r["kind"] == "oracle" and r["unit"] == "tokens/s" and r["value"] > 0
        assert 1 <= r["cores"] <= w.H and "initial state" in r["sample"]
