"""Tensor-core prefill parity: the tcgen05 kernel against the fp64 oracle, at
small sizes that span many chunks and ragged tails, and at the full size of
the bf16 batch workload on sampled chains.

Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
(liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle

from _helpers import (TOL_BF16_FRO, TOL_BF16_MAXN, assert_close, oracle_prefill, rel_fro, to_np)
from hybrid_linear_attention_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def watchdog(kda):
    lib = kda.load()
    flags = ctypes.c_uint(0)
    lib.kda_device_watchdog.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.c_int]
    assert lib.kda_device_watchdog(ctypes.byref(flags), 1) == 0
    return flags.value


def run(kda, x, kernel="tc", **kw):
    o, s = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["initial_state"],
                             x["cu_seqlens"], kernel=kernel, **kw)
    torch.cuda.synchronize()
    return o, s


@pytest.fixture(autouse=True)
def _no_timeouts(kda):
    watchdog(kda)
    yield
    assert watchdog(kda) == 0, "a tensor-core kernel wait ran out"


@pytest.mark.parametrize("lens", [[64], [1], [65, 63, 200], [1000, 3, 0, 129]])
def test_tc_matches_oracle(kda, lens):
    w = inputs.scaled(inputs.VARLEN_64, H=3)
    x = inputs.make_prefill(w, device=DEV, lengths=np.array(lens))
    o, s = run(kda, x)
    o_ref, s_ref = oracle_prefill(x)
    assert_close(to_np(o), o_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="o")
    assert_close(to_np(s), s_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="S")


def test_tc_zero_initial_state(kda):
    w = inputs.scaled(inputs.PREFILL_B4_T8K, B=2, T=300, H=2)
    x = inputs.make_prefill(w, device=DEV)
    x["cu_seqlens"] = None
    o, s = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, None, kernel="tc", B=2)
    torch.cuda.synchronize()
    x["cu_seqlens"] = torch.tensor([0, 300, 600], dtype=torch.int32, device=DEV)
    o_ref, s_ref = oracle_prefill(x)
    assert_close(to_np(o), o_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="o")
    assert_close(to_np(s), s_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="S")


def test_tc_agrees_with_simt(kda):
    """Both kernels compute the same chunk form; their bf16 rounding differs."""
    w = inputs.scaled(inputs.VARLEN_64, H=4)
    x = inputs.make_prefill(w, device=DEV, lengths=np.array([777, 64, 5]))
    o1, s1 = run(kda, x, kernel="tc")
    o2, s2 = run(kda, x, kernel="simt")
    assert rel_fro(to_np(o1), to_np(o2)) <= 1e-2
    assert rel_fro(to_np(s1), to_np(s2)) <= 1e-2


@pytest.mark.parametrize("pattern", ["all_floor", "one_channel", "alternating"])
def test_tc_range_guard(kda, pattern):
    """g at the floor of [K3-notes §2.2, Eq. 5] in every pattern that sends a
    chunk down the four-round (per 16-token tile) Gram path."""
    w = inputs.scaled(inputs.VARLEN_64, H=2)
    x = inputs.make_prefill(w, device=DEV, lengths=np.array([300, 130]))
    g = x["log_alpha"]
    if pattern == "all_floor":
        g.fill_(-5.0)
    elif pattern == "one_channel":
        g[:, :, 77] = -5.0
    else:
        g[0:64] = -5.0
        g[128:192] = -5.0
        g[310:374] = -5.0
    o, s = run(kda, x)
    assert torch.isfinite(o.float()).all() and torch.isfinite(s).all()
    o_ref, s_ref = oracle_prefill(x)
    assert_close(to_np(o), o_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="o")
    assert_close(to_np(s), s_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="S")


def test_tc_exact_recall_in_chunk(kda):
    """beta = 1, q = k one-hot keys: every token reads back its own v inside the
    chunk, which needs A's diagonal ([K3-notes §2.2]) and the UT transform."""
    N, T, H, d = 1, 256, 2, 128
    gen = torch.Generator(device=DEV).manual_seed(3)
    idx = torch.randint(0, d, (T, H), generator=gen, device=DEV)
    k = torch.zeros(T, H, d, device=DEV).scatter_(2, idx[..., None], 1.0).to(torch.bfloat16)
    v = torch.randn(T, H, d, generator=gen, device=DEV).to(torch.bfloat16)
    g = -torch.rand(T, H, d, generator=gen, device=DEV) * 0.5
    beta = torch.ones(T, H, device=DEV)
    o, _ = kda.kda_chunk_fwd(k.clone(), k, v, g, beta, None, None, kernel="tc")
    torch.cuda.synchronize()
    assert rel_fro(to_np(o), to_np(v)) <= 1e-2


def test_tc_full_size_batch_workload_sampled(kda):
    """The bf16 batch workload at full size (B=4, H=32, T=8192, d=128, C=64),
    in the launch configuration the benchmark times; the oracle checks 6
    (sequence, head) chains end to end."""
    w = inputs.PREFILL_B4_T8K
    x = inputs.make_prefill(w, device=DEV)
    o, s = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, None, B=w.B)
    torch.cuda.synchronize()
    chains = [0, 37, 64 + 5, 96 + 31, 3 * 32 + 16, 31]
    rows = {c: (slice((c // w.H) * w.T, (c // w.H + 1) * w.T), c % w.H) for c in chains}
    # host copies of just the sampled heads keep the oracle call small
    o_ref, s_ref = oracle_prefill(x, chains=chains)
    for c in chains:
        sl, h = rows[c]
        n = c // w.H
        assert_close(to_np(o[sl, h]), o_ref[sl, h], TOL_BF16_FRO, TOL_BF16_MAXN, what=f"o chain {c}")
        assert_close(to_np(s[n, h]), s_ref[n, h], TOL_BF16_FRO, TOL_BF16_MAXN, what=f"S chain {c}")


def test_tc_full_size_varlen_workload_sampled(kda):
    """The packed varlen workload at full size (64 sequences of 512..32768
    tokens, H=32, random initial states), run as the benchmark runs it; the
    oracle checks the chains of the shortest and the longest sequence and of
    four others."""
    w = inputs.VARLEN_64
    x = inputs.make_prefill(w, device=DEV)
    o, s = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["initial_state"],
                             x["cu_seqlens"])
    torch.cuda.synchronize()
    lens = np.asarray(x["lengths"])
    seqs = [int(np.argmin(lens)), int(np.argmax(lens)), 1, 17, 40, 63]
    heads = [0, 31, 5, 12, 20, 27]
    cu = x["cu_seqlens"].cpu().numpy()
    for n, h in zip(seqs, heads):
        # the chain alone (one sequence, one head) keeps the host copies small
        sl = slice(int(cu[n]), int(cu[n + 1]))
        hs = slice(h, h + 1)
        sub = {name: inputs.host_f32(x[name][sl, hs].contiguous()) for name in ("q", "k", "v", "log_alpha", "beta")}
        s0 = inputs.host_f32(x["initial_state"][n:n + 1, hs].contiguous())
        o_ref, s_ref = oracle.recurrent(sub["q"], sub["k"], sub["v"], sub["log_alpha"], sub["beta"], s0)
        assert_close(to_np(o[sl, hs]), o_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what=f"o seq {n} head {h}")
        assert_close(to_np(s[n:n + 1, hs]), s_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what=f"S seq {n} head {h}")


def test_tc_deterministic_and_resume(kda):
    w = inputs.scaled(inputs.PREFILL_B4_T8K, B=1, T=3000, H=2, random_initial_state=True)
    x = inputs.make_prefill(w, device=DEV)
    x["cu_seqlens"] = None
    o1, s1 = run(kda, x)
    o2, s2 = run(kda, x)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    cut = 2560
    pa = {n: x[n][:cut].contiguous() for n in ("q", "k", "v", "log_alpha", "beta")}
    pb = {n: x[n][cut:].contiguous() for n in ("q", "k", "v", "log_alpha", "beta")}
    oa, sa = run(kda, {**pa, "initial_state": x["initial_state"], "cu_seqlens": None})
    ob, sb = run(kda, {**pb, "initial_state": sa, "cu_seqlens": None})
    assert torch.equal(torch.cat([oa, ob]), o1) and torch.equal(sb, s1)


@pytest.mark.parametrize("nseq", [512, 600])
def test_tc_many_packed_sequences(kda, nseq):
    """Packed batches of many short sequences, ragged and empty ones among them:
    up to 512 sequences each work item ranks the lengths and runs the sequences
    longest first; beyond that it keeps index order.  Either way every
    (sequence, head) chain must match the oracle and land in its own rows and
    final-state slot."""
    rng = np.random.default_rng(nseq)
    lens = rng.integers(0, 140, size=nseq)
    lens[::37] = 0
    lens[5] = 257  # one long sequence that is not first in index order
    w = inputs.scaled(inputs.VARLEN_64, H=2)
    x = inputs.make_prefill(w, device=DEV, lengths=lens)
    o, s = run(kda, x)
    o_ref, s_ref = oracle_prefill(x)
    assert_close(to_np(o), o_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="o")
    assert_close(to_np(s), s_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="S")


@pytest.mark.parametrize("decay", ["workload", "alternating_floor"])
def test_tc_split_and_plain_orders_agree_bitwise(kda, decay):
    """The kernel runs its state group in one of two orders, chosen at launch:
    with at most one (sequence, head) chain per SM, V~'s first half and its
    M5/M6 overlap M7's last steps; otherwise the plain order.  Both form the
    same products with the same accumulation order, so B=5 x H=32 chains
    (more than the SMs: plain) and their first 4 sequences alone (128 chains:
    split) give bitwise equal outputs and states, ragged last chunk and
    (with the alternating floor) the per-tile range path included.  The
    batch is also checked against the oracle on a few chains."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    w = inputs.scaled(inputs.PREFILL_B4_T8K, B=5, T=300, random_initial_state=True)
    assert w.B * w.H > sms >= (w.B - 1) * w.H
    x = inputs.make_prefill(w, device=DEV)
    if decay == "alternating_floor":
        x["log_alpha"].view(w.B, w.T, w.H, w.dk)[:, 64:128] = -5.0
    o5, s5 = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["initial_state"], None,
                               B=w.B)
    n4 = (w.B - 1) * w.T
    sub = {n: x[n][:n4].contiguous() for n in ("q", "k", "v", "log_alpha", "beta")}
    o4, s4 = kda.kda_chunk_fwd(sub["q"], sub["k"], sub["v"], sub["log_alpha"], sub["beta"],
                               x["initial_state"][: w.B - 1].contiguous(), None, B=w.B - 1)
    torch.cuda.synchronize()
    assert torch.equal(o4, o5[:n4]) and torch.equal(s4, s5[: w.B - 1])
    chains = [0, 33, 4 * 32 + 7]
    o_ref, s_ref = oracle_prefill(x, chains=chains)
    for c in chains:
        n, h = divmod(c, w.H)
        sl = slice(n * w.T, (n + 1) * w.T)
        assert_close(to_np(o5[sl, h]), o_ref[sl, h], TOL_BF16_FRO, TOL_BF16_MAXN, what=f"o chain {c}")
        assert_close(to_np(s5[n, h]), s_ref[n, h], TOL_BF16_FRO, TOL_BF16_MAXN, what=f"S chain {c}")
