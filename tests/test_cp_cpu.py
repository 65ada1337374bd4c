"""The multi-rank context-parallel schedule (kda_chunk_fwd_cp) on CPU ranks.

Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
(liuzhao09.github.io/papers/kimi-k3), [K3-notes] below: §2.5, the
context-parallel affine pair.

Two and three gloo ranks each hold one contiguous token segment of every
sequence and run the library's schedule (pair, one all-gather, composition,
local rerun) with the fp64 oracle as the compute: what is checked is the
schedule itself (which segment's pair goes where, the composition order,
rank 0's initial state reaching every rank, the last rank holding the final
state) against the oracle's single run of the whole sequences.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleBackend:
    """The schedule's three compute steps by the oracle, on CPU tensors."""

    pair_dtype = torch.float64

    def affine_pair(self, q, k, v, g, beta, B):
        import oracle
        L = q.shape[0] // B
        H, dk, dv = q.shape[1], q.shape[2], v.shape[2]
        out = torch.zeros(2, B, H, dk, dv, dtype=torch.float64)
        for n in range(B):
            sl = slice(n * L, (n + 1) * L)
            for h in range(H):
                M, St = oracle.affine_pair(k[sl].numpy(), v[sl].numpy(), g[sl].numpy(), beta[sl].numpy(), h, 0, L)
                out[0, n, h] = torch.from_numpy(St)
                out[1, n, h] = torch.from_numpy(M)
        return out

    def compose(self, pairs, s0):
        # E_0 = s0, E_{p+1} = S~_p + M_p E_p, for every sequence and head
        _, B, Pm1, H, dk, dv = pairs.shape
        E = torch.zeros(B, Pm1 + 1, H, dk, dv, dtype=torch.float64)
        E[:, 0] = s0
        for p in range(Pm1):
            E[:, p + 1] = pairs[0, :, p] + torch.matmul(pairs[1, :, p], E[:, p])
        return E

    def forward(self, q, k, v, g, beta, entry, B):
        import oracle
        L = q.shape[0] // B
        cu = np.arange(B + 1) * L
        o, s = oracle.recurrent(q.numpy(), k.numpy(), v.numpy(), g.numpy(), beta.numpy(),
                                None if entry is None else entry.numpy(), cu)
        return torch.from_numpy(o), torch.from_numpy(s)


def make_problem(B=2, T=24, H=2, d=4, seed=7):
    rng = np.random.default_rng(seed)
    f = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))  # noqa: E731
    q = rng.standard_normal((B * T, H, d))
    k = rng.standard_normal((B * T, H, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B * T, H, d))
    g = rng.uniform(np.log(0.5), -1e-3, (B * T, H, d))
    beta = 1 / (1 + np.exp(-rng.standard_normal((B * T, H))))
    s0 = torch.from_numpy(rng.standard_normal((B, H, d, d)) * 0.3)
    return f(q), f(k), f(v), f(g), f(beta), s0


def shard(x, B, T, rank, world):
    L = T // world
    return torch.cat([x[n * T + rank * L: n * T + (rank + 1) * L] for n in range(B)], 0).contiguous()


def _rank_main(rank, world, port, results, B, T):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    sys.path.insert(0, os.path.join(root, "tests"))
    import torch.distributed as dist
    from hybrid_linear_attention_chunk_gb300.cp import kda_chunk_fwd_cp, torch_all_gather
    from test_cp_cpu import OracleBackend, make_problem, shard
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v, g, beta, s0 = make_problem(B=B, T=T)
        loc = [shard(x, B, T, rank, world) for x in (q, k, v, g, beta)]
        o, s = kda_chunk_fwd_cp(*loc, s0 if rank == 0 else None, rank=rank, world=world, B=B,
                                all_gather=torch_all_gather(), backend=OracleBackend())
        results[rank] = (o.numpy(), s.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_cp_schedule_on_gloo_ranks_matches_one_run(world):
    import oracle
    B, T = 2, 24
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, results, B, T), nprocs=world, join=True)
        res = dict(results)
    q, k, v, g, beta, s0 = make_problem(B=B, T=T)
    o_ref, s_ref = oracle.recurrent(q.numpy(), k.numpy(), v.numpy(), g.numpy(), beta.numpy(), s0.numpy(),
                                    np.arange(B + 1) * T)
    L = T // world
    for r in range(world):
        o_r, s_r = res[r]
        want = np.concatenate([o_ref[n * T + r * L: n * T + (r + 1) * L] for n in range(B)], 0)
        assert np.allclose(o_r, want, rtol=1e-10, atol=1e-12), f"rank {r} outputs"
    assert np.allclose(res[world - 1][1], s_ref, rtol=1e-10, atol=1e-12), "final state on the last rank"


def test_single_rank_is_the_plain_call():
    import oracle
    from hybrid_linear_attention_chunk_gb300.cp import kda_chunk_fwd_cp
    q, k, v, g, beta, s0 = make_problem(B=1, T=10)
    o, s = kda_chunk_fwd_cp(q, k, v, g, beta, s0, rank=0, world=1, B=1, backend=OracleBackend())
    o_ref, s_ref = oracle.recurrent(q.numpy(), k.numpy(), v.numpy(), g.numpy(), beta.numpy(), s0.numpy())
    assert np.array_equal(o.numpy(), o_ref) and np.array_equal(s.numpy(), s_ref)


def _bench_rank_main(rank, world, port, results):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    sys.path.insert(0, os.path.join(root, "tests"))
    import torch.distributed as dist
    import bench
    from hybrid_linear_attention_chunk_gb300 import inputs
    from test_cp_cpu import OracleBackend
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = inputs.scaled(inputs.LONG_T1M, T=48, H=2, dk=8, dv=8, qkv_dtype=torch.float32,
                          out_dtype=torch.float32)
        results[rank] = bench.time_cp(None, inputs, 2, torch.device("cpu"), world, rank, w=w,
                                      backend=OracleBackend())
    finally:
        dist.destroy_process_group()


def test_bench_cp_leg_on_gloo_ranks():
    """bench.py's context-parallel leg (run under torchrun with N > 1): every
    rank times the same schedule on its token segment, and the line carries
    every rank's time, the max over ranks and the bytes each rank sends."""
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_bench_rank_main, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    for r in range(world):
        e = res[r]
        assert e["path"] == "kda_chunk_fwd_cp" and e["ranks"] == world and e["tokens_per_rank"] == 24
        assert len(e["per_rank_ms"]) == world and e["per_rank_ms"] == res[0]["per_rank_ms"]
        assert e["ms_per_step"] == round(max(e["per_rank_ms"]), 3) and e["ms_per_step"] > 0
        assert e["allgather_bytes_per_rank"] == 3 * 1 * 2 * 8 * 8 * 4
        assert e["scaling"] == "strong" and e["tokens_per_s"] > 0
