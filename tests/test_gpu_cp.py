"""Long sequences split into segments joined through their affine pairs
([K3-notes §2.5, context-parallel affine pair]), against the fp64 oracle and
against the unsplit tensor-core kernel.

Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
(liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.
"""
import numpy as np
import pytest
import torch

from _helpers import (TOL_BF16_FRO, TOL_BF16_MAXN, assert_close, max_norm, oracle_heads_by_columns,
                      oracle_prefill, rel_fro, to_np)
from hybrid_linear_attention_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run(kda, x, B, **kw):
    o, s = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["initial_state"], None,
                             B=B, **kw)
    torch.cuda.synchronize()
    return o, s


def long_inputs(B, T, H, seed_index=2):
    w = inputs.scaled(inputs.LONG_T1M, B=B, T=T, H=H)
    return w, inputs.make_prefill(w, device=DEV)


@pytest.mark.parametrize("T,segments", [(4096, 4), (4000, 3), (1000, 7)])
def test_segments_match_oracle(kda, T, segments):
    w, x = long_inputs(2, T, 2)
    o, s = run(kda, x, 2, segments=segments)
    o_ref, s_ref = oracle_prefill(x)
    assert_close(to_np(o), o_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="o")
    assert_close(to_np(s), s_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="S")


def test_segments_agree_with_unsplit(kda):
    w, x = long_inputs(1, 8192, 3)
    o1, s1 = run(kda, x, 1, segments=1)
    o4, s4 = run(kda, x, 1, segments=5)
    assert rel_fro(to_np(o4), to_np(o1)) <= 1e-2
    assert rel_fro(to_np(s4), to_np(s1)) <= 1e-2


def test_caller_workspace_equals_stream_ordered(kda):
    w, x = long_inputs(1, 3000, 2)
    d = kda.chunk_desc(x["q"], x["v"], gate_dtype=0, segments=4, B=1)
    nbytes = kda.kda_chunk_fwd_workspace_size(d)
    assert nbytes == (3 * 4 - 5) * 1 * 2 * 128 * 128 * 4  # P-2 pairs and P-1 entry states per chain
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    o1, s1 = run(kda, x, 1, segments=4)
    o2, s2 = run(kda, x, 1, segments=4, workspace=ws)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    small = torch.empty(nbytes - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(kda.KdaError) as e:
        run(kda, x, 1, segments=4, workspace=small)
    assert e.value.status == -2


def test_split_refused_where_unsupported(kda):
    w = inputs.scaled(inputs.VARLEN_64, H=2)
    x = inputs.make_prefill(w, device=DEV, lengths=np.array([300, 200]))
    with pytest.raises(kda.KdaError) as e:
        kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["initial_state"],
                          x["cu_seqlens"], segments=2)
    assert e.value.status == -7


def test_long_context_full_size(kda):
    """The long-context workload at full size (B=1, H=16, T=1,048,576, slow
    decay, random initial state ~ N(0, 0.02)).  The automatic plan splits it
    into segments joined through their affine pairs ([K3-notes §2.5]).

    * Heads 0 and 11 against the fp64 oracle over all 2^20 tokens: every
      output row, checked in 16 consecutive slices of the sequence (so every
      segment and every segment join is covered, the last segment included),
      and the final state.
    * Every head's final state and a strided sample of every head's outputs
      against the unsplit kernel."""
    w = inputs.LONG_T1M
    x = inputs.make_prefill(w, device=DEV)
    d = kda.chunk_desc(x["q"], x["v"], gate_dtype=0, B=1)
    assert kda.kda_chunk_fwd_workspace_size(d) > 0  # the planner splits this shape
    o_cp, s_cp = run(kda, x, 1)
    assert torch.isfinite(o_cp.float()).all() and torch.isfinite(s_cp).all()
    heads = [0, 11]
    o_ref, s_ref = oracle_heads_by_columns(x, heads)
    got_o = o_cp[:, heads]
    for i, h in enumerate(heads):
        assert_close(to_np(s_cp[:, h]), s_ref[:, i], TOL_BF16_FRO, TOL_BF16_MAXN, what=f"final state head {h}")
        for sl in range(16):
            r0, r1 = sl * w.T // 16, (sl + 1) * w.T // 16
            assert_close(to_np(got_o[r0:r1, i]), o_ref[r0:r1, i], TOL_BF16_FRO, TOL_BF16_MAXN,
                         what=f"o head {h} rows [{r0}, {r1})")
    del o_ref, s_ref, got_o
    o_1, s_1 = run(kda, x, 1, segments=1)
    assert rel_fro(to_np(s_cp), to_np(s_1)) <= 1e-2
    rows = torch.arange(0, w.T, 97, device=DEV)
    assert rel_fro(to_np(o_cp[rows]), to_np(o_1[rows])) <= 1e-2


# ----------------------------------------------- context parallelism across ranks

def _shard(t, B, T, rank, world):
    L = T // world
    return torch.cat([t[n * T + rank * L: n * T + (rank + 1) * L] for n in range(B)], 0).contiguous()


@pytest.mark.parametrize("world", [2, 4])
def test_cp_ranks_emulated_in_sequence(kda, world):
    """The multi-GPU schedule (kda_chunk_fwd_cp) with the library on this GPU,
    its ranks run one after another; the all-gather hands every rank the
    stack of what all ranks send (each rank's own send is checked against
    it).  Outputs and the last rank's final state match the oracle."""
    from hybrid_linear_attention_chunk_gb300.cp import LibraryBackend, kda_chunk_fwd_cp
    w = inputs.scaled(inputs.LONG_T1M, B=2, T=4096, H=2)
    x = inputs.make_prefill(w, device=DEV)
    B, T = w.B, w.T
    names = ("q", "k", "v", "log_alpha", "beta")
    shards = [[_shard(x[nm], B, T, r, world) for nm in names] for r in range(world)]
    backend = LibraryBackend(kda)
    sends = []
    for r in range(world):
        pair = (backend.affine_pair(*shards[r], B) if r < world - 1
                else torch.zeros(2, B, w.H, w.dk, w.dv, device=DEV))
        s0 = x["initial_state"] if r == 0 else torch.zeros_like(pair[0])
        sends.append(torch.cat([pair, s0[None]], 0))
    stacked = torch.stack(sends)

    def gather_for(r):
        def gather(t):
            assert torch.equal(t, stacked[r]), f"rank {r} sent something else"
            return stacked
        return gather

    outs, state = [], None
    for r in range(world):
        o, s = kda_chunk_fwd_cp(*shards[r], x["initial_state"] if r == 0 else None, rank=r, world=world, B=B,
                                all_gather=gather_for(r), backend=backend)
        outs.append(o)
        state = s
    torch.cuda.synchronize()
    L = T // world
    o_full = torch.empty(B * T, w.H, w.dv, dtype=outs[0].dtype, device=DEV)
    for r in range(world):
        for n in range(B):
            o_full[n * T + r * L: n * T + (r + 1) * L] = outs[r][n * L:(n + 1) * L]
    o_ref, s_ref = oracle_prefill(x)
    assert_close(to_np(o_full), o_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="o")
    assert_close(to_np(state), s_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="final state")


def test_affine_pair_and_compose_match_the_segmented_plan(kda):
    """The two CP entry points on one GPU: the pair of the first half and the
    composed entry state of the second half give the same final state as the
    unsplit call, within bf16 tolerance."""
    w = inputs.scaled(inputs.LONG_T1M, B=1, T=2048, H=3)
    x = inputs.make_prefill(w, device=DEV)
    first = {nm: x[nm][:1024].contiguous() for nm in ("q", "k", "v", "log_alpha", "beta")}
    second = {nm: x[nm][1024:].contiguous() for nm in ("q", "k", "v", "log_alpha", "beta")}
    pairs = kda.kda_chunk_affine_pair(first["q"], first["k"], first["v"], first["log_alpha"], first["beta"], B=1)
    E = kda.kda_affine_compose(pairs[:, :, None].contiguous(), x["initial_state"])
    o2, s2 = kda.kda_chunk_fwd(second["q"], second["k"], second["v"], second["log_alpha"], second["beta"],
                               E[:, 1].contiguous(), None, B=1)
    o, s = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["initial_state"], None, B=1,
                             segments=1)
    torch.cuda.synchronize()
    assert torch.equal(E[:, 0], x["initial_state"])
    assert_close(to_np(s2), to_np(s), TOL_BF16_FRO, TOL_BF16_MAXN, what="final state")
    assert_close(to_np(o2), to_np(o[1024:]), TOL_BF16_FRO, TOL_BF16_MAXN, what="second half o")


def test_nccl_all_gather_single_rank(kda):
    """The schedule's all-gather through NCCL on a one-rank group."""
    import socket

    import torch.distributed as dist
    from hybrid_linear_attention_chunk_gb300.cp import torch_all_gather
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        t = torch.arange(24, dtype=torch.float32, device=DEV).reshape(2, 3, 4)
        got = torch_all_gather()(t)
        torch.cuda.synchronize()
        assert got.shape == (1, 2, 3, 4) and torch.equal(got[0], t)
    finally:
        dist.destroy_process_group()
