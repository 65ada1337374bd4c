"""Seeded synthetic inputs for the KDA workloads.

This module is the one piece shared by the CUDA path's tests/bench and by the
oracle's callers.  It draws random numbers and casts them; it holds none of
the recurrence's arithmetic.

Workloads (the distributions follow the five synthetic workloads this library
is measured on; all seeded):

* q, k ~ N(0, 1), L2-normalised per (token, head) in fp32, then cast to the
  input dtype with round-to-nearest-even; v ~ N(0, 1) cast the same way.
* log_alpha ~ U[ln 0.5, -1e-3] per channel (long-context workload:
  U[ln 0.9, -1e-4]); beta = sigmoid(N(0, 1)); both fp32.
* initial state ~ N(0, 0.02) read as standard deviation 0.02, fp32.
* varlen lengths: floor(exp(U[ln 512, ln 32768])).

Draw order per workload: q, k, v, log_alpha, beta, initial state, lengths.
Generation runs with torch's generator on the requested device (CPU for the
small workloads in tests, the GPU for the full-size ones, where host
generation would take minutes).  The oracle always receives the same tensors,
copied to the host, so both sides see identical values.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

SEED_BASE = 20260000


@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    T: int
    H: int
    dk: int
    dv: int
    chunk: int
    qkv_dtype: torch.dtype
    out_dtype: torch.dtype
    g_lo: float
    g_hi: float
    random_initial_state: bool
    varlen_seqs: int = 0          # >0: packed varlen with this many sequences
    len_lo: int = 512
    len_hi: int = 32768
    seed_index: int = 0


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    N: int
    H: int
    dk: int
    dv: int
    steps: int
    qkv_dtype: torch.dtype
    out_dtype: torch.dtype
    g_lo: float
    g_hi: float
    seed_index: int = 3


LN05 = math.log(0.5)
LN09 = math.log(0.9)

# The five synthetic workloads, indexed as the seeds are (SEED_BASE + index).
TINY_FP32 = PrefillWorkload("tiny_fp32_B1_H2_T256_d64_C64", 1, 256, 2, 64, 64, 64,
                            torch.float32, torch.float32, LN05, -1e-3, False, seed_index=0)
PREFILL_B4_T8K = PrefillWorkload("prefill_bf16_B4_H32_T8192_d128_C64", 4, 8192, 32, 128, 128, 64,
                                 torch.bfloat16, torch.bfloat16, LN05, -1e-3, False, seed_index=1)
LONG_T1M = PrefillWorkload("prefill_bf16_B1_H16_T1048576_d128_C64", 1, 1 << 20, 16, 128, 128, 64,
                           torch.bfloat16, torch.bfloat16, LN09, -1e-4, True, seed_index=2)
DECODE_N256 = DecodeWorkload("decode_N256_H32_d128_1000steps", 256, 32, 128, 128, 1000,
                             torch.bfloat16, torch.bfloat16, LN05, -1e-3, seed_index=3)
VARLEN_64 = PrefillWorkload("varlen_bf16_64seqs_len512to32768_H32_d128_C64", 1, 0, 32, 128, 128, 64,
                            torch.bfloat16, torch.bfloat16, LN05, -1e-3, True, varlen_seqs=64,
                            seed_index=4)

WORKLOADS = {w.name: w for w in (TINY_FP32, PREFILL_B4_T8K, LONG_T1M, DECODE_N256, VARLEN_64)}


def scaled(w: PrefillWorkload, **kw) -> PrefillWorkload:
    """A copy of workload w with some fields replaced (used for small test sizes)."""
    return dataclasses.replace(w, **kw)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    # L2 normalisation of the last axis in fp32: a property of the synthetic
    # input distribution, not a step of the library (which never normalises).
    return x / torch.linalg.vector_norm(x, dim=-1, keepdim=True).clamp_min(1e-30)


def varlen_lengths(num_seqs: int, lo: int, hi: int, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    u = rng.uniform(math.log(lo), math.log(hi), size=num_seqs)
    return np.floor(np.exp(u)).astype(np.int64)


def make_prefill(w: PrefillWorkload, device="cpu", seed: Optional[int] = None,
                 lengths: Optional[np.ndarray] = None) -> dict:
    """Inputs for one prefill workload.

    Returns a dict with q, k [T_total,H,dk], v [T_total,H,dv] (w.qkv_dtype),
    log_alpha [T_total,H,dk] fp32, beta [T_total,H] fp32, initial_state
    [N,H,dk,dv] fp32 or None, cu_seqlens int32 [N+1], and N, T_total.
    The [B,T,H,d] layout of a batch is viewed as B packed sequences of T.
    """
    seed = SEED_BASE + w.seed_index if seed is None else seed
    if w.varlen_seqs > 0:
        if lengths is None:
            lengths = varlen_lengths(w.varlen_seqs, w.len_lo, w.len_hi, seed)
        lengths = np.asarray(lengths, dtype=np.int64)
    else:
        lengths = np.full(w.B, w.T, dtype=np.int64)
    N = len(lengths)
    cu = np.zeros(N + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    Tt = int(cu[-1])
    gen = _gen(device, seed)
    H, dk, dv = w.H, w.dk, w.dv
    q = _unit_rows(torch.randn(Tt, H, dk, generator=gen, device=device)).to(w.qkv_dtype)
    k = _unit_rows(torch.randn(Tt, H, dk, generator=gen, device=device)).to(w.qkv_dtype)
    v = torch.randn(Tt, H, dv, generator=gen, device=device).to(w.qkv_dtype)
    g = torch.rand(Tt, H, dk, generator=gen, device=device) * (w.g_hi - w.g_lo) + w.g_lo
    beta = torch.sigmoid(torch.randn(Tt, H, generator=gen, device=device))
    s0 = None
    if w.random_initial_state:
        s0 = torch.randn(N, H, dk, dv, generator=gen, device=device) * 0.02
    return dict(q=q, k=k, v=v, log_alpha=g.contiguous(), beta=beta.contiguous(),
                initial_state=s0, cu_seqlens=torch.from_numpy(cu.astype(np.int32)).to(device),
                N=N, T_total=Tt, lengths=lengths)


def make_decode(w: DecodeWorkload, steps: int, device="cpu", seed: Optional[int] = None) -> dict:
    """Inputs for `steps` consecutive decode steps: q, k [steps,N,H,dk], v
    [steps,N,H,dv], log_alpha [steps,N,H,dk], beta [steps,N,H] and the fp32
    state [N,H,dk,dv] ~ N(0, 0.02)."""
    seed = SEED_BASE + w.seed_index if seed is None else seed
    gen = _gen(device, seed)
    N, H, dk, dv = w.N, w.H, w.dk, w.dv
    q = _unit_rows(torch.randn(steps, N, H, dk, generator=gen, device=device)).to(w.qkv_dtype)
    k = _unit_rows(torch.randn(steps, N, H, dk, generator=gen, device=device)).to(w.qkv_dtype)
    v = torch.randn(steps, N, H, dv, generator=gen, device=device).to(w.qkv_dtype)
    g = torch.rand(steps, N, H, dk, generator=gen, device=device) * (w.g_hi - w.g_lo) + w.g_lo
    beta = torch.sigmoid(torch.randn(steps, N, H, generator=gen, device=device))
    s0 = torch.randn(N, H, dk, dv, generator=gen, device=device) * 0.02
    return dict(q=q, k=k, v=v, log_alpha=g, beta=beta, state=s0)


def make_layer_gates(rows: int, H: int, dk: int, dv: int, dtype: torch.dtype, device="cpu",
                     seed: int = SEED_BASE + 100, z_mean: float = -3.0, z_std: float = 1.5) -> dict:
    """Gate inputs of the KDA layer form for `rows` tokens (or decode rows).

    z (decay logits) [rows,H,dk] ~ N(z_mean, z_std^2) and out_gate [rows,H,dv]
    ~ N(0, 1), cast to `dtype`; A_log [H] ~ U[-0.5, 0.5] and norm_weight [dv]
    ~ U[0.5, 1.5] in fp32.  With the default z the per-channel decays spread
    from close to 1 to a few percent per token (most chunks keep one decay
    reference); z_mean = 3 puts most channels near the Eq. 5 floor, where
    every chunk takes the per-tile path.  Draw order: z, out_gate, A_log,
    norm_weight.
    """
    gen = _gen(device, seed)
    z = (torch.randn(rows, H, dk, generator=gen, device=device) * z_std + z_mean).to(dtype)
    og = torch.randn(rows, H, dv, generator=gen, device=device).to(dtype)
    A = torch.rand(H, generator=gen, device=device) - 0.5
    w = torch.rand(dv, generator=gen, device=device) + 0.5
    return dict(z=z.contiguous(), out_gate=og.contiguous(), A_log=A.contiguous(), norm_weight=w.contiguous())


def host_f32(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """Exact float32 copy on the host (bf16 upcasts exactly)."""
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float32).numpy()
