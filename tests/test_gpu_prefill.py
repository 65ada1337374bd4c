"""Prefill parity: libkda.so (through its C ABI) against the fp64 oracle.

Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
(liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.
"""
import dataclasses

import numpy as np
import pytest
import torch

from _helpers import (TOL_BF16_FRO, TOL_BF16_MAXN, TOL_F32_FRO, assert_close, oracle_prefill, to_np)
from hybrid_linear_attention_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run(kda, x, chunk=64, kernel="auto", **kw):
    o, s = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["initial_state"],
                             x["cu_seqlens"], chunk=chunk, kernel=kernel, **kw)
    torch.cuda.synchronize()
    return o, s


def check(o, s, o_ref, s_ref, fp32, what="", rows=None):
    o_n = to_np(o)
    if rows is not None:
        o_n, o_ref = o_n[rows], o_ref[rows]
    if fp32:
        assert_close(o_n, o_ref, TOL_F32_FRO, what=what + " o")
        assert_close(to_np(s), s_ref, TOL_F32_FRO, what=what + " S")
    else:
        assert_close(o_n, o_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what=what + " o")
        assert_close(to_np(s), s_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what=what + " S")


def test_tiny_fp32_workload(kda):
    """B=1, H=2, T=256, d=64, C=64, fp32 everywhere, zero initial state."""
    x = inputs.make_prefill(inputs.TINY_FP32, device=DEV)
    o, s = run(kda, x)
    o_ref, s_ref = oracle_prefill(x)
    check(o, s, o_ref, s_ref, fp32=True, what="tiny fp32")


@pytest.mark.parametrize("C", [16, 32, 64])
@pytest.mark.parametrize("dk,dv", [(16, 32), (64, 64), (128, 128), (32, 128)])
def test_simt_shapes_fp32(kda, C, dk, dv):
    w = inputs.scaled(inputs.TINY_FP32, H=3, dk=dk, dv=dv, chunk=C, random_initial_state=True,
                      varlen_seqs=3, len_lo=1, len_hi=200)
    x = inputs.make_prefill(w, device=DEV, lengths=np.array([1, 150, 2 * C + 3]))
    o, s = run(kda, x, chunk=C, kernel="simt")
    o_ref, s_ref = oracle_prefill(x)
    check(o, s, o_ref, s_ref, fp32=True, what=f"simt C={C} dk={dk} dv={dv}")


@pytest.mark.parametrize("kernel", ["simt", "auto"])
def test_bf16_varlen_ragged_with_states(kda, kernel):
    w = inputs.scaled(inputs.VARLEN_64, H=4)
    x = inputs.make_prefill(w, device=DEV, lengths=np.array([300, 1, 64, 0, 129, 700]))
    o, s = run(kda, x, kernel=kernel)
    o_ref, s_ref = oracle_prefill(x)
    check(o, s, o_ref, s_ref, fp32=False, what=f"bf16 varlen {kernel}")


@pytest.mark.parametrize("kernel", ["simt", "auto"])
def test_decay_floor_everywhere(kda, kernel):
    """g = -5 on every channel (the floor of [K3-notes §2.2, Eq. 5]): the
    cumulative log-decay of a 64-token chunk reaches -320, which the range
    guard has to handle without overflow."""
    w = inputs.scaled(inputs.VARLEN_64, H=2)
    x = inputs.make_prefill(w, device=DEV, lengths=np.array([200, 77]))
    x["log_alpha"].fill_(-5.0)
    o, s = run(kda, x, kernel=kernel)
    assert torch.isfinite(o.float()).all() and torch.isfinite(s).all()
    o_ref, s_ref = oracle_prefill(x)
    check(o, s, o_ref, s_ref, fp32=False, what=f"g=-5 {kernel}")


@pytest.mark.parametrize("kernel", ["simt", "auto"])
def test_mixed_fast_and_guarded_chunks(kda, kernel):
    """Chunks at the floor next to ordinary chunks, and a single channel at
    the floor, so that fast and guarded chunks alternate within a sequence."""
    w = inputs.scaled(inputs.VARLEN_64, H=2)
    x = inputs.make_prefill(w, device=DEV, lengths=np.array([400]))
    g = x["log_alpha"]
    g[64:128] = -5.0
    g[200:264, :, 7] = -5.0
    o, s = run(kda, x, kernel=kernel)
    o_ref, s_ref = oracle_prefill(x)
    check(o, s, o_ref, s_ref, fp32=False, what=f"mixed {kernel}")


def test_fp32_decay_floor(kda):
    w = inputs.scaled(inputs.TINY_FP32, T=200, random_initial_state=True)
    x = inputs.make_prefill(w, device=DEV)
    x["log_alpha"][:, 0].fill_(-5.0)
    o, s = run(kda, x)
    o_ref, s_ref = oracle_prefill(x)
    check(o, s, o_ref, s_ref, fp32=True, what="fp32 g=-5 head 0")


def test_chunk_size_invariance_fp32(kda):
    """Outputs do not depend on the chunk length beyond rounding."""
    w = inputs.scaled(inputs.TINY_FP32, T=333, H=2, random_initial_state=True)
    x = inputs.make_prefill(w, device=DEV)
    outs = [run(kda, x, chunk=C) for C in (16, 32, 64)]
    for o, s in outs[1:]:
        assert torch.allclose(o, outs[0][0], atol=2e-5, rtol=1e-4)
        assert torch.allclose(s, outs[0][1], atol=2e-5, rtol=1e-4)


def _slice(x, a, b, s0):
    y = {n: x[n][a:b].contiguous() for n in ("q", "k", "v", "log_alpha", "beta")}
    y.update(initial_state=s0, cu_seqlens=None)
    return y


@pytest.mark.parametrize("kernel", ["simt", "auto"])
def test_resume_equals_single_run(kda, kernel):
    """Prefix-cache resume ([K3-notes §2.5, Fig. 12], resume boundary B = 2560):
    [0, B) then [B, T) from the saved final state equals one pass over [0, T)."""
    T, Bs = 3000, 2560
    w = inputs.scaled(inputs.PREFILL_B4_T8K, B=1, T=T, H=2, random_initial_state=True)
    x = inputs.make_prefill(w, device=DEV)
    x["cu_seqlens"] = None
    o_full, s_full = run(kda, x, kernel=kernel)
    o1, s1 = run(kda, _slice(x, 0, Bs, x["initial_state"]), kernel=kernel)
    o2, s2 = run(kda, _slice(x, Bs, T, s1), kernel=kernel)
    x["cu_seqlens"] = torch.tensor([0, T], dtype=torch.int32, device=DEV)
    o_ref, s_ref = oracle_prefill(x)
    check(torch.cat([o1, o2]), s2, o_ref, s_ref, fp32=False, what="resume")
    # Bs is a multiple of 64, so the chunk boundaries coincide: bitwise equal
    assert torch.equal(torch.cat([o1, o2]), o_full) and torch.equal(s2, s_full)


@pytest.mark.parametrize("kernel", ["simt", "auto"])
def test_varlen_equals_separate_calls_bitwise(kda, kernel):
    w = inputs.scaled(inputs.VARLEN_64, H=2)
    lens = np.array([130, 64, 5])
    x = inputs.make_prefill(w, device=DEV, lengths=lens)
    o, s = run(kda, x, kernel=kernel)
    cu = np.concatenate([[0], np.cumsum(lens)])
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        xn = _slice(x, cu[n], cu[n + 1], x["initial_state"][n:n + 1].contiguous())
        on, sn = run(kda, xn, kernel=kernel)
        assert torch.equal(on, o[sl]) and torch.equal(sn[0], s[n])


@pytest.mark.parametrize("kernel", ["simt", "auto"])
def test_deterministic(kda, kernel):
    w = inputs.scaled(inputs.VARLEN_64, H=4)
    x = inputs.make_prefill(w, device=DEV, lengths=np.array([500, 77]))
    o1, s1 = run(kda, x, kernel=kernel)
    o2, s2 = run(kda, x, kernel=kernel)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_padding_tokens_are_identity(kda):
    """Tokens with g = 0, beta = 0 and k = 0 leave the state as it was, the
    same fact the kernels use to pad a ragged last chunk."""
    w = inputs.scaled(inputs.TINY_FP32, T=100, random_initial_state=True)
    x = inputs.make_prefill(w, device=DEV)
    for n in ("log_alpha", "beta", "k"):
        x[n][40:].zero_()
    _, s_full = run(kda, x)
    _, s_40 = run(kda, _slice(x, 0, 40, x["initial_state"]))
    assert torch.allclose(s_full, s_40, atol=1e-6, rtol=1e-5)


def test_validate_mode_reports_out_of_range(kda):
    w = inputs.scaled(inputs.TINY_FP32, T=64)
    x = inputs.make_prefill(w, device=DEV)
    run(kda, x, validate=True)  # in range: fine
    x["log_alpha"][3, 1, 5] = -6.0
    with pytest.raises(kda.KdaError) as e:
        run(kda, x, validate=True)
    assert e.value.status == -5
    x["log_alpha"][3, 1, 5] = -1.0
    x["beta"][7, 0] = 1.5
    with pytest.raises(kda.KdaError):
        run(kda, x, validate=True)


def test_validate_mode_rejects_bad_cu_seqlens(kda):
    w = inputs.scaled(inputs.VARLEN_64, H=2)
    x = inputs.make_prefill(w, device=DEV, lengths=np.array([10, 20]))
    x["cu_seqlens"][1] = 31  # cu = [0, 31, 30]: decreasing
    with pytest.raises(kda.KdaError) as e:
        run(kda, x, validate=True)
    assert e.value.status == -5


def test_tc_request_on_unsupported_shape_is_an_error(kda):
    x = inputs.make_prefill(inputs.TINY_FP32, device=DEV)  # fp32: not a tensor-core shape
    with pytest.raises(kda.KdaError) as e:
        run(kda, x, kernel="tc")
    assert e.value.status == -7


def test_empty_sequences_keep_initial_state(kda):
    w = inputs.scaled(inputs.VARLEN_64, H=2)
    x = inputs.make_prefill(w, device=DEV, lengths=np.array([0, 3, 0]))
    o, s = run(kda, x)
    assert torch.equal(s[0], x["initial_state"][0]) and torch.equal(s[2], x["initial_state"][2])
