"""Context parallelism across GPUs for long sequences.

Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
(liuzhao09.github.io/papers/kimi-k3), [K3-notes] below: §2.5, the
context-parallel affine pair.  A segment of a sequence maps any entry state
to S_out = S~ + M S_in; the pairs are a fixed size whatever the segment's
length, so R ranks that each hold one contiguous segment of every sequence
exchange only their pairs:

  1. pair_r  = affine pair of the local segment          (library kernel)
  2. all-gather of the R pairs                           (the one collective)
  3. E_r     = entry state of segment r, composed from pairs 0..r-1 and the
               initial state held by rank 0              (library kernel)
  4. out_r, S_r = the local segment from E_r             (library kernel)

Rank R-1's final state is the sequences' final state.  This module only
orders the steps and moves the pairs; the arithmetic runs in libkda.  The
compute steps and the all-gather are parameters so that the same schedule
can run on CPU ranks in tests.
"""
from __future__ import annotations

from typing import Callable, Optional

import torch


class LibraryBackend:
    """The compute steps on this rank's GPU through libkda."""

    pair_dtype = torch.float32  # every rank sends the same dtype and shape

    def __init__(self, kda_module):
        self.kda = kda_module

    def affine_pair(self, q, k, v, log_alpha, beta, B):
        return self.kda.kda_chunk_affine_pair(q, k, v, log_alpha, beta, B=B)

    def compose(self, pairs, initial_state):
        return self.kda.kda_affine_compose(pairs, initial_state)

    def forward(self, q, k, v, log_alpha, beta, entry_state, B):
        return self.kda.kda_chunk_fwd(q, k, v, log_alpha, beta, entry_state, None, B=B)


def torch_all_gather(group=None) -> Callable[[torch.Tensor], torch.Tensor]:
    """all-gather through torch.distributed (NCCL on GPUs, gloo on CPUs):
    returns a function mapping this rank's tensor to the [R, ...] stack."""
    import torch.distributed as dist

    def gather(t: torch.Tensor) -> torch.Tensor:
        world = dist.get_world_size(group)
        t = t.contiguous()
        if t.is_cuda:
            out = torch.empty((world,) + tuple(t.shape), dtype=t.dtype, device=t.device)
            dist.all_gather_into_tensor(out, t, group=group)
            return out
        parts = [torch.empty_like(t) for _ in range(world)]
        dist.all_gather(parts, t, group=group)
        return torch.stack(parts)

    return gather


def kda_chunk_fwd_cp(q, k, v, log_alpha, beta, initial_state=None, *, rank: int, world: int, B: int,
                     all_gather: Optional[Callable] = None, backend=None):
    """kda_chunk_fwd of B sequences split over `world` ranks by tokens.

    This rank holds tokens [rank L, (rank + 1) L) of every sequence: q, k,
    log_alpha [B*L, H, dk], v [B*L, H, dv], beta [B*L, H] (B sequences of L
    tokens each, sequence-major).  initial_state [B, H, dk, dv] is read on rank
    0 only (None: zero).  Returns (out for the local tokens, the state after
    the local segment); on rank world-1 that state is the final state.
    """
    if backend is None:
        from . import _lib
        backend = LibraryBackend(_lib)
    if world == 1:
        return backend.forward(q, k, v, log_alpha, beta, initial_state, B)
    if all_gather is None:
        all_gather = torch_all_gather()
    H, dk, dv = q.shape[-2], q.shape[-1], v.shape[-1]
    # what this rank sends: its pair (the last rank's is never used: zeros)
    # and, from rank 0, the initial state, so that one all-gather carries all
    if rank < world - 1:
        pair = backend.affine_pair(q, k, v, log_alpha, beta, B)
    else:
        pair = torch.zeros(2, B, H, dk, dv, dtype=backend.pair_dtype, device=q.device)
    s0 = initial_state if (rank == 0 and initial_state is not None) else torch.zeros_like(pair[0])
    gathered = all_gather(torch.cat([pair, s0.to(pair.dtype)[None]], 0))   # [world, 3, B, H, dk, dv]
    before = gathered[: world - 1, :2].permute(1, 2, 0, 3, 4, 5).contiguous()  # [2, B, world-1, H, dk, dv]
    entries = backend.compose(before, gathered[0, 2].contiguous())           # [B, world, H, dk, dv]
    return backend.forward(q, k, v, log_alpha, beta, entries[:, rank].contiguous(), B)
