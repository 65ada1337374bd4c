"""The KDA layer form (kda_layer_fwd, kda_layer_decode_step) against the fp64
oracle's ``layer`` / ``layer_decode_step``: log-decay formed in the kernels
from decay logits, and the per-head RMSNorm with the sigmoid output gate.

Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
(liuzhao09.github.io/papers/kimi-k3), [K3-notes] below (§2.2, Eq. 5 and the
KDA output equation).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from _helpers import TOL_BF16_FRO, TOL_BF16_MAXN, TOL_F32_FRO, assert_close, to_np
from hybrid_linear_attention_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def oracle_layer(x, gt, with_gate, eps):
    h = {n: inputs.host_f32(x[n]) for n in ("q", "k", "v", "beta", "initial_state")}
    cu = x["cu_seqlens"].cpu().numpy().astype(np.int64)
    return oracle.layer(h["q"], h["k"], h["v"], inputs.host_f32(gt["z"]), h["beta"], inputs.host_f32(gt["A_log"]),
                        -5.0, out_gate=inputs.host_f32(gt["out_gate"]) if with_gate else None,
                        norm_weight=inputs.host_f32(gt["norm_weight"]) if with_gate else None, norm_eps=eps,
                        initial_state=h["initial_state"], cu_seqlens=cu)


def assert_y_close(y, x, gt, eps, fro, maxn, what="y"):
    """y against the oracle, each row scaled back by the oracle's RMS of o.

    RMSNorm divides a row by its RMS, so an absolute error d in o becomes
    d / rms(o) in y.  The kernels' error in o is bounded against the sizes of
    the terms that sum to it (bf16 operands), not against the row's own RMS, so
    a row whose terms cancel (fast decay and a small k.q) has a large relative
    error after the norm however good o is.  Scaling both rows by the same
    positive factor rms(o_ref) measures y in o's units; a wrong norm factor,
    gate or weight still shows at full size."""
    o_ref, _ = oracle_layer(x, gt, False, eps)
    y_ref, _ = oracle_layer(x, gt, True, eps)
    rms = np.sqrt(np.mean(o_ref ** 2, axis=-1, keepdims=True) + eps)
    assert_close(to_np(y) * rms, y_ref * rms, fro, maxn, what=what)
    return y_ref


def run_layer(kda, x, gt, with_gate, eps, **kw):
    return kda.kda_layer_fwd(x["q"], x["k"], x["v"], gt["z"], x["beta"], gt["A_log"], -5.0,
                             out_gate=gt["out_gate"] if with_gate else None,
                             norm_weight=gt["norm_weight"] if with_gate else None, norm_eps=eps,
                             initial_state=x["initial_state"], cu_seqlens=x["cu_seqlens"], **kw)


@pytest.mark.parametrize("kernel", ["tc", "simt"])
@pytest.mark.parametrize("with_gate", [True, False])
@pytest.mark.parametrize("z_mean", [-3.0, 3.0])
def test_layer_packed_sequences(kda, kernel, with_gate, z_mean):
    """Packed ragged sequences (one empty) with a random initial state; z_mean
    3 drives most channels to the decay floor (the per-tile range path)."""
    lens = np.array([300, 0, 128, 700, 64, 513])
    if kernel == "tc":
        w, fro, maxn = inputs.scaled(inputs.VARLEN_64, H=2), TOL_BF16_FRO, TOL_BF16_MAXN
    else:
        w = inputs.scaled(inputs.TINY_FP32, H=2, varlen_seqs=len(lens), random_initial_state=True)
        fro, maxn = TOL_F32_FRO, None
    x = inputs.make_prefill(w, device=DEV, lengths=lens)
    gt = inputs.make_layer_gates(x["T_total"], w.H, w.dk, w.dv, w.qkv_dtype, device=DEV, z_mean=z_mean)
    eps = 1e-6
    o, s = run_layer(kda, x, gt, with_gate, eps, kernel=kernel, validate=True)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle_layer(x, gt, with_gate, eps)
    if with_gate:
        assert_y_close(o, x, gt, eps, fro, maxn)
    else:
        assert_close(to_np(o), o_ref, fro, maxn, what="o")
    assert_close(to_np(s), s_ref, fro, maxn, what="S")


def test_layer_batch_segments_and_tails(kda):
    """A B x T batch on the tensor-core kernel, unsplit and split into three
    segments (the gate applies in every pass; the output gate only where the
    output is written), with a ragged tail of 37 tokens per sequence."""
    w = dataclasses.replace(inputs.PREFILL_B4_T8K, B=2, T=1600 + 37, H=2)
    x = inputs.make_prefill(w, device=DEV)
    gt = inputs.make_layer_gates(x["T_total"], w.H, w.dk, w.dv, w.qkv_dtype, device=DEV)
    _, s_ref = oracle_layer(x, gt, True, 1e-5)
    for seg in (1, 3):
        o, s = kda.kda_layer_fwd(x["q"], x["k"], x["v"], gt["z"], x["beta"], gt["A_log"], -5.0,
                                 out_gate=gt["out_gate"], norm_weight=gt["norm_weight"], norm_eps=1e-5,
                                 kernel="tc", segments=seg, B=w.B)
        torch.cuda.synchronize()
        assert_y_close(o, x, gt, 1e-5, TOL_BF16_FRO, TOL_BF16_MAXN, what=f"y segments={seg}")
        assert_close(to_np(s), s_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what=f"S segments={seg}")


def test_layer_equals_chunk_fwd_on_the_gate_decay(kda):
    """Without the output gate, the layer call is kda_chunk_fwd fed the
    log-decay that Eq. 5 gives (formed here in fp32 by torch) within rounding."""
    lens = np.array([640, 200])
    w = inputs.scaled(inputs.VARLEN_64, H=2)
    x = inputs.make_prefill(w, device=DEV, lengths=lens)
    gt = inputs.make_layer_gates(x["T_total"], w.H, w.dk, w.dv, w.qkv_dtype, device=DEV)
    o1, s1 = run_layer(kda, x, gt, False, 0.0)
    g = -5.0 * torch.sigmoid(torch.exp(gt["A_log"])[None, :, None] * gt["z"].float())
    o2, s2 = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], g.contiguous(), x["beta"], x["initial_state"],
                               x["cu_seqlens"])
    torch.cuda.synchronize()
    assert_close(to_np(s1), to_np(s2), 2e-3, what="S")
    assert_close(to_np(o1), to_np(o2), 1e-2, what="o")


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float32)])
@pytest.mark.parametrize("with_gate", [True, False])
def test_layer_decode_step(kda, d, dtype, with_gate):
    w = dataclasses.replace(inputs.DECODE_N256, N=6, H=3, dk=d, dv=d, qkv_dtype=dtype, out_dtype=dtype)
    x = inputs.make_decode(w, steps=3, device=DEV)
    gt = inputs.make_layer_gates(3 * w.N, w.H, d, d, dtype, device=DEV)
    z = gt["z"].view(3, w.N, w.H, d)
    og = gt["out_gate"].view(3, w.N, w.H, d)
    S = x["state"].clone()
    S_ref = inputs.host_f32(x["state"]).astype(np.float64)
    fro = TOL_F32_FRO if dtype == torch.float32 else TOL_BF16_FRO
    for t in range(3):
        o = kda.kda_layer_decode_step(x["q"][t], x["k"][t], x["v"][t], z[t].contiguous(), x["beta"][t], S,
                                      gt["A_log"], -5.0, out_gate=og[t].contiguous() if with_gate else None,
                                      norm_weight=gt["norm_weight"] if with_gate else None, norm_eps=1e-6,
                                      validate=True)
        torch.cuda.synchronize()
        o_ref, S_ref = oracle.layer_decode_step(
            *(inputs.host_f32(x[n][t]) for n in ("q", "k", "v")), inputs.host_f32(z[t]),
            inputs.host_f32(x["beta"][t]), S_ref, inputs.host_f32(gt["A_log"]), -5.0,
            out_gate=inputs.host_f32(og[t]) if with_gate else None,
            norm_weight=inputs.host_f32(gt["norm_weight"]) if with_gate else None, norm_eps=1e-6)
        assert_close(to_np(o), o_ref, fro, what=f"y step {t}")
        assert_close(to_np(S), S_ref, 1e-5, what=f"S step {t}")


def test_layer_validate_rejects_bad_values(kda):
    w = inputs.scaled(inputs.VARLEN_64, H=2)
    x = inputs.make_prefill(w, device=DEV, lengths=np.array([128, 64]))
    gt = inputs.make_layer_gates(x["T_total"], w.H, w.dk, w.dv, w.qkv_dtype, device=DEV)
    z = gt["z"].clone()
    z[5, 1, 7] = float("nan")
    with pytest.raises(kda.KdaError) as e:
        kda.kda_layer_fwd(x["q"], x["k"], x["v"], z, x["beta"], gt["A_log"], cu_seqlens=x["cu_seqlens"],
                          validate=True)
    assert e.value.status == -5
    A = gt["A_log"].clone()
    A[1] = float("inf")
    with pytest.raises(kda.KdaError) as e:
        kda.kda_layer_fwd(x["q"], x["k"], x["v"], gt["z"], x["beta"], A, cu_seqlens=x["cu_seqlens"],
                          validate=True)
    assert e.value.status == -5
    with pytest.raises(kda.KdaError) as e:   # a floor below Eq. 5's -5 is refused without validate
        kda.kda_layer_fwd(x["q"], x["k"], x["v"], gt["z"], x["beta"], gt["A_log"], g_min=-5.5,
                          cu_seqlens=x["cu_seqlens"])
    assert e.value.status == -5


def test_layer_many_chains_plain_and_split_orders_agree(kda):
    """Decay logits without the output gate, on more (sequence, head) chains
    than the GPU has SMs (80 packed sequences x 2 heads: the plain
    state-group order) against the oracle, and the first 8 of those sequences
    alone (16 chains: the split order) bitwise equal to their rows of the
    large call.  Lengths 1..200, so most sequences end in a ragged chunk."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(11)
    lens = rng.integers(1, 201, size=80)
    w = inputs.scaled(inputs.VARLEN_64, H=2)
    assert len(lens) * w.H > sms
    x = inputs.make_prefill(w, device=DEV, lengths=lens)
    gt = inputs.make_layer_gates(x["T_total"], w.H, w.dk, w.dv, w.qkv_dtype, device=DEV)
    o, s = run_layer(kda, x, gt, False, 0.0, kernel="tc")
    o_ref, s_ref = oracle_layer(x, gt, False, 0.0)
    torch.cuda.synchronize()
    assert_close(to_np(o), o_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="o")
    assert_close(to_np(s), s_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="S")
    k = 8
    cu = x["cu_seqlens"].cpu().numpy()
    end = int(cu[k])
    sub = {n: x[n][:end].contiguous() for n in ("q", "k", "v", "beta")}
    sub["initial_state"] = x["initial_state"][:k].contiguous()
    sub["cu_seqlens"] = x["cu_seqlens"][: k + 1].contiguous()
    gsub = {"z": gt["z"][:end].contiguous(), "A_log": gt["A_log"]}
    o8, s8 = run_layer(kda, sub, gsub, False, 0.0, kernel="tc")
    torch.cuda.synchronize()
    assert torch.equal(o8, o[:end]) and torch.equal(s8, s[:k])
