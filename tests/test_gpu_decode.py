"""Decode-step parity: libkda.so (through its C ABI) against the fp64 oracle.

Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
(liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from _helpers import (TOL_BF16_FRO, TOL_BF16_MAXN, assert_close, max_norm, oracle_prefill, rel_fro,
                      to_np)
from hybrid_linear_attention_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def step_host(dx, t):
    return [inputs.host_f32(dx[n][t]) for n in ("q", "k", "v", "log_alpha", "beta")]


@pytest.mark.parametrize("N,H,dk,dv", [(4, 3, 128, 128), (3, 2, 64, 64), (2, 2, 16, 128),
                                      (5, 1, 128, 32)])
@pytest.mark.parametrize("qkv", [torch.bfloat16, torch.float32])
def test_decode_steps_match_oracle(kda, N, H, dk, dv, qkv):
    w = dataclasses.replace(inputs.DECODE_N256, N=N, H=H, dk=dk, dv=dv, qkv_dtype=qkv, out_dtype=qkv)
    steps = 20
    dx = inputs.make_decode(w, steps=steps, device=DEV)
    st = dx["state"].clone()
    s_ref = inputs.host_f32(dx["state"]).astype(np.float64)
    for t in range(steps):
        o = kda.kda_decode_step(dx["q"][t], dx["k"][t], dx["v"][t], dx["log_alpha"][t], dx["beta"][t], st)
        o_ref, s_ref = oracle.decode_step(*step_host(dx, t), s_ref)
        tol = 1e-4 if qkv == torch.float32 else TOL_BF16_FRO
        assert_close(to_np(o), o_ref, tol, what=f"o step {t}")
    torch.cuda.synchronize()
    # the state is fp32 in both dtypes; only rounding of fp32 arithmetic differs
    assert rel_fro(to_np(st), s_ref) <= 1e-5


def test_decode_full_width_sampled(kda):
    """The decode workload's full size (N=256, H=32, d=128, fp32 state
    [256,32,128,128] ~ N(0, 0.02)) for a few steps, every output and a sample
    of 64 states checked."""
    w = inputs.DECODE_N256
    steps = 3
    dx = inputs.make_decode(w, steps=steps, device=DEV)
    st = dx["state"].clone()
    rng = np.random.default_rng(0)
    chains = np.sort(rng.choice(w.N * w.H, 64, replace=False)).astype(np.int32)
    s_ref = inputs.host_f32(dx["state"]).astype(np.float64)
    for t in range(steps):
        o = kda.kda_decode_step(dx["q"][t], dx["k"][t], dx["v"][t], dx["log_alpha"][t], dx["beta"][t], st)
        o_ref, s_ref = oracle.decode_step(*step_host(dx, t), s_ref)
        assert_close(to_np(o), o_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what=f"o step {t}")
    s_gpu = to_np(st).reshape(w.N * w.H, w.dk, w.dv)[chains]
    s_ref = s_ref.reshape(w.N * w.H, w.dk, w.dv)[chains]
    assert rel_fro(s_gpu, s_ref) <= 1e-5


def test_decode_steps_equal_prefill(kda):
    """T decode steps from S_0 give the same outputs and state as one prefill
    of those T tokens from S_0 (both forms of [K3-notes §2.2])."""
    N, H, T = 3, 2, 70
    w = dataclasses.replace(inputs.DECODE_N256, N=N, H=H)
    dx = inputs.make_decode(w, steps=T, device=DEV)
    st = dx["state"].clone()
    outs = []
    for t in range(T):
        outs.append(kda.kda_decode_step(dx["q"][t], dx["k"][t], dx["v"][t], dx["log_alpha"][t],
                                        dx["beta"][t], st))
    o_dec = torch.stack(outs)  # [T, N, H, dv]
    # prefill layout: sequence n is tokens [n*T, (n+1)*T)
    perm = lambda a: a.transpose(0, 1).reshape(N * T, *a.shape[2:]).contiguous()
    q, k, v, g = (perm(dx[n]) for n in ("q", "k", "v", "log_alpha"))
    beta = perm(dx["beta"])
    o_pre, s_pre = kda.kda_chunk_fwd(q, k, v, g, beta, dx["state"].contiguous(), None, B=N)
    torch.cuda.synchronize()
    o_dec = o_dec.transpose(0, 1).reshape(N * T, H, -1)
    assert rel_fro(to_np(st), to_np(s_pre)) <= 2e-2
    assert rel_fro(to_np(o_dec), to_np(o_pre)) <= 2e-2


def test_decode_exact_recall(kda):
    """beta = 1, q = k with |k| = 1 returns v_t whatever the state
    ([K3-notes §2.2]: erase along k, then write)."""
    N, H, d = 8, 4, 128
    g = torch.Generator(device=DEV).manual_seed(5)
    k = torch.zeros(N, H, d, device=DEV)
    idx = torch.randint(0, d, (N, H), generator=g, device=DEV)
    k.scatter_(2, idx[..., None], 1.0)  # one-hot keys: unit norm exactly
    v = torch.randn(N, H, d, generator=g, device=DEV)
    la = -torch.rand(N, H, d, generator=g, device=DEV)
    beta = torch.ones(N, H, device=DEV)
    st = torch.randn(N, H, d, d, generator=g, device=DEV)
    o = kda.kda_decode_step(k.clone(), k, v, la, beta, st)
    torch.cuda.synchronize()
    assert torch.allclose(o, v, atol=1e-5, rtol=1e-5)


def test_decode_validate_mode(kda):
    w = dataclasses.replace(inputs.DECODE_N256, N=2, H=2)
    dx = inputs.make_decode(w, steps=1, device=DEV)
    st = dx["state"].clone()
    kda.kda_decode_step(dx["q"][0], dx["k"][0], dx["v"][0], dx["log_alpha"][0], dx["beta"][0], st,
                        validate=True)
    bad = dx["beta"][0].clone()
    bad[1, 1] = -0.1
    with pytest.raises(kda.KdaError) as e:
        kda.kda_decode_step(dx["q"][0], dx["k"][0], dx["v"][0], dx["log_alpha"][0], bad, st,
                            validate=True)
    assert e.value.status == -5


def test_decode_workload_all_1000_steps(kda):
    """The decode workload as stated: N=256, H=32, d=128, fp32 state
    ~ N(0, 0.02), 1000 consecutive steps from the workload's seed.

    * 64 fixed (sequence, head) pairs follow the oracle's own trajectory
      through all 1000 steps: every output at every step, and the state at
      steps 9, 99 and 999.
    * Every head at steps 0..9 against the oracle's full trajectory (all
      8192 heads), and every head at steps 99 and 999 against one oracle step
      taken from the library's state just before that step.

    o is bf16 (tolerances rel-Frobenius 2e-2, max-normalised 5e-2).  The
    state is fp32 on both sides from identical inputs, so only fp32 rounding
    separates them: with per-channel decays below 1 the state forgets old
    rounding errors, and after 1000 steps a rel-Frobenius of 1e-4 is far
    above what ~1000 fp32 roundings of ~6e-8 can add up to ([K3-notes §2.2]:
    the recurrence is non-expansive for unit keys and beta in [0, 1])."""
    w = inputs.DECODE_N256
    steps = w.steps
    assert steps == 1000
    dx = inputs.make_decode(w, steps=steps, device=DEV)
    st = dx["state"].clone()
    N, H, dk, dv = w.N, w.H, w.dk, w.dv
    rng = np.random.default_rng(0)
    chains = np.sort(rng.choice(N * H, 64, replace=False))
    n_idx = torch.as_tensor(chains // H, device=DEV)
    h_idx = torch.as_tensor(chains % H, device=DEV)
    names = ("q", "k", "v", "log_alpha", "beta")
    # the sampled pairs' inputs for all steps, as 64 single-head sequences
    sub = {nm: inputs.host_f32(dx[nm][:, n_idx, h_idx]) for nm in names}
    s_sub = inputs.host_f32(dx["state"][n_idx, h_idx]).astype(np.float64)[:, None]
    s_all = inputs.host_f32(dx["state"]).astype(np.float64)
    o_sub = torch.empty(steps, 64, dv, dtype=dx["v"].dtype, device=DEV)
    full_from_gpu = {99, 999}
    state_checks = {9, 99, 999}
    worst = [0.0, 0.0]
    for t in range(steps):
        prev = to_np(st).astype(np.float64) if t in full_from_gpu else None
        o = kda.kda_decode_step(dx["q"][t], dx["k"][t], dx["v"][t], dx["log_alpha"][t], dx["beta"][t], st)
        o_sub[t] = o[n_idx, h_idx]
        # the sampled pairs through the oracle's own trajectory
        ins = [sub[nm][t][:, None] for nm in names]
        o_ref, s_sub = oracle.decode_step(*ins, s_sub)
        if t < 10:  # every head, the oracle's full trajectory
            o_all, s_all = oracle.decode_step(*step_host(dx, t), s_all)
            assert_close(to_np(o), o_all, TOL_BF16_FRO, TOL_BF16_MAXN, what=f"o all heads step {t}")
            if t == 9:
                assert rel_fro(to_np(st), s_all) <= 1e-4, "state of every head after step 9"
        if prev is not None:  # every head, one oracle step from the library's state
            o1, s1 = oracle.decode_step(*step_host(dx, t), prev)
            assert_close(to_np(o), o1, TOL_BF16_FRO, TOL_BF16_MAXN, what=f"o all heads step {t}")
            assert rel_fro(to_np(st), s1) <= 1e-5, f"state of every head after step {t} (one step)"
        if t in state_checks:
            s_gpu = to_np(st[n_idx, h_idx]).astype(np.float64)
            e = rel_fro(s_gpu, s_sub[:, 0])
            assert e <= 1e-4, f"sampled states after step {t}: rel-Frobenius {e:.2e}"
            assert_close(s_gpu, s_sub[:, 0], TOL_BF16_FRO, TOL_BF16_MAXN, what=f"sampled states step {t}")
        o_sub_ref = o_ref[:, 0]
        got = to_np(o_sub[t])
        worst[0] = max(worst[0], rel_fro(got, o_sub_ref))
        worst[1] = max(worst[1], max_norm(got, o_sub_ref))
    assert worst[0] <= TOL_BF16_FRO and worst[1] <= TOL_BF16_MAXN, f"sampled outputs: worst {worst}"
