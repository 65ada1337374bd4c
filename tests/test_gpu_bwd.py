"""Backward of the chunked prefill (kda_chunk_bwd) against the fp64 oracle's
reverse-mode gradients (``oracle.backward``), which are pinned to finite
differences of the forward recurrence.

Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
(liuzhao09.github.io/papers/kimi-k3), [K3-notes] below (§2.2: the chunkwise
form is the training form).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_close, to_np
from hybrid_linear_attention_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
# The backward computes in fp32 from the exact input values (bf16 inputs are
# read exactly), so fp32 tolerances apply to every workload.
TOL = 1e-4


def upstream(x, w, dtype, seed=77):
    gen = torch.Generator(device=DEV)
    gen.manual_seed(seed)
    dO = torch.randn(x["T_total"], w.H, w.dv, generator=gen, device=DEV).to(dtype)
    dST = torch.randn(x["N"], w.H, w.dk, w.dv, generator=gen, device=DEV) * 0.1
    return dO, dST


def oracle_grads(x, dO, dST):
    h = {n: inputs.host_f32(x[n]) for n in ("q", "k", "v", "log_alpha", "beta", "initial_state")}
    cu = x["cu_seqlens"].cpu().numpy().astype(np.int64)
    return oracle.backward(h["q"], h["k"], h["v"], h["log_alpha"], h["beta"], inputs.host_f32(dO),
                           initial_state=h["initial_state"], d_final_state=inputs.host_f32(dST), cu_seqlens=cu)


def check(gr, ref, what=""):
    for name, rname in (("dq", "dq"), ("dk", "dk"), ("dv", "dv"), ("dlog_alpha", "dg"), ("dbeta", "dbeta"),
                        ("d_initial_state", "ds0")):
        assert_close(to_np(gr[name]), ref[rname], TOL, what=f"{what} {name}")


@pytest.mark.parametrize("wl", ["fp32_d64", "bf16_d128"])
def test_bwd_packed_sequences(kda, wl):
    """Packed ragged sequences, one empty, with initial states and a final-state gradient."""
    lens = np.array([37, 0, 16, 100, 5])
    if wl == "fp32_d64":
        w = inputs.scaled(inputs.TINY_FP32, H=2, varlen_seqs=len(lens), random_initial_state=True)
    else:
        w = inputs.scaled(inputs.VARLEN_64, H=2)
    x = inputs.make_prefill(w, device=DEV, lengths=lens)
    dO, dST = upstream(x, w, w.out_dtype)
    gr = kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], dO, x["initial_state"], dST,
                           x["cu_seqlens"], validate=True)
    torch.cuda.synchronize()
    check(gr, oracle_grads(x, dO, dST), wl)


def test_bwd_batch_fast_decay(kda):
    """A B x T batch (no cu_seqlens, zero initial state, no final-state gradient)
    with log-decay down to the -5 floor: every 16-token chunk stays in range."""
    w = dataclasses.replace(inputs.PREFILL_B4_T8K, B=2, T=300, H=3, g_lo=-5.0, g_hi=-0.5)
    x = inputs.make_prefill(w, device=DEV)
    dO, _ = upstream(x, w, w.out_dtype)
    gr = kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], dO, B=w.B)
    torch.cuda.synchronize()
    ref = oracle_grads(x, dO, torch.zeros(x["N"], w.H, w.dk, w.dv, device=DEV))
    check(gr, ref, "batch")


def test_bwd_long_sequences_and_workspace(kda):
    """Two 2000-token sequences with a caller workspace; the same call again
    gives bitwise the same gradients."""
    lens = np.array([2000, 1984])
    w = inputs.scaled(inputs.VARLEN_64, H=2)
    x = inputs.make_prefill(w, device=DEV, lengths=lens)
    dO, dST = upstream(x, w, w.out_dtype, seed=5)
    d = kda.chunk_desc(x["q"], x["v"], cu_seqlens=x["cu_seqlens"], out_dtype=dO.dtype, gate_dtype=0)
    ws = torch.empty(kda.kda_chunk_bwd_workspace_size(d), dtype=torch.uint8, device=DEV)
    args = (x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], dO, x["initial_state"], dST, x["cu_seqlens"])
    g1 = kda.kda_chunk_bwd(*args, workspace=ws)
    g1 = {k: v.clone() for k, v in g1.items()}
    g2 = kda.kda_chunk_bwd(*args, workspace=ws)
    torch.cuda.synchronize()
    for name in g1:
        assert torch.equal(g1[name], g2[name]), name
    check(g1, oracle_grads(x, dO, dST), "long")


def test_bwd_matches_forward_differences(kda):
    """A directional derivative through the library itself: with a random
    direction u for the log-decay, (L(g + e u) - L(g - e u)) / 2e from two
    fp32 forward calls (fp32 workload) agrees with <dlog_alpha, u>."""
    lens = np.array([70, 45])
    w = inputs.scaled(inputs.TINY_FP32, H=2, varlen_seqs=2, random_initial_state=True)
    x = inputs.make_prefill(w, device=DEV, lengths=lens)
    dO, dST = upstream(x, w, torch.float32, seed=9)
    gr = kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], dO, x["initial_state"], dST,
                           x["cu_seqlens"])
    gen = torch.Generator(device=DEV)
    gen.manual_seed(3)
    u = torch.randn(x["log_alpha"].shape, generator=gen, device=DEV) * 0.05

    def L(g):
        o, s = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], g.contiguous(), x["beta"], x["initial_state"],
                                 x["cu_seqlens"], kernel="simt")
        return float((o.double() * dO.double()).sum() + (s.double() * dST.double()).sum())

    eps = 1e-2
    fd = (L(x["log_alpha"] + eps * u) - L(x["log_alpha"] - eps * u)) / (2 * eps)
    an = float((gr["dlog_alpha"].double() * u.double()).sum())
    assert abs(fd - an) <= 2e-3 * max(abs(an), 1.0), (fd, an)


@pytest.mark.parametrize("dk,dv", [(32, 16), (16, 64), (16, 16), (128, 32), (64, 128)])
def test_bwd_shapes_fp32(kda, dk, dv):
    """Other head sizes (the scans' 16-column tiling at dv = 16; at dk = dv = 16
    the scans' dk split leaves two channels per thread group, below one 128-bit
    load; at dk = 16 one warp holds all gradient channels), packed ragged
    sequences."""
    lens = np.array([50, 17, 33])
    w = inputs.scaled(inputs.TINY_FP32, H=3, dk=dk, dv=dv, varlen_seqs=len(lens), random_initial_state=True)
    x = inputs.make_prefill(w, device=DEV, lengths=lens)
    dO, dST = upstream(x, w, torch.float32, seed=dk + dv)
    gr = kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], dO, x["initial_state"], dST,
                           x["cu_seqlens"])
    torch.cuda.synchronize()
    check(gr, oracle_grads(x, dO, dST), f"dk={dk} dv={dv}")
