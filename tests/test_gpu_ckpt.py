"""State checkpoints during prefill (kda_chunk_fwd_ckpt) against the fp64
oracle's recorded states, on both prefill kernels, packed and batched inputs
and the segmented long-sequence plan; and prefix-cache resume through the
library: continuing from a checkpoint reproduces the full run.

Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
(liuzhao09.github.io/papers/kimi-k3), [K3-notes] below (§2.5, Fig. 12).
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import TOL_BF16_FRO, TOL_BF16_MAXN, TOL_F32_FRO, assert_close, to_np
from hybrid_linear_attention_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def oracle_ckpt(x, every):
    h = {n: inputs.host_f32(x[n]) for n in ("q", "k", "v", "log_alpha", "beta", "initial_state")}
    cu = x["cu_seqlens"].cpu().numpy().astype(np.int64)
    return oracle.recurrent_ckpt(h["q"], h["k"], h["v"], h["log_alpha"], h["beta"], every,
                                 initial_state=h["initial_state"], cu_seqlens=cu)


def cu_ckpt_for(x, every):
    lens = np.diff(x["cu_seqlens"].cpu().numpy())
    c = np.concatenate([[0], np.cumsum(lens // every)]).astype(np.int32)
    return torch.from_numpy(c).to(DEV)


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_ckpt_packed_sequences(kda, kernel):
    every = 128
    lens = np.array([300, 0, 128, 700, 64, 513])
    if kernel == "tc":
        w, fro, maxn = inputs.scaled(inputs.VARLEN_64, H=2), TOL_BF16_FRO, TOL_BF16_MAXN
    else:
        w, fro, maxn = inputs.scaled(inputs.TINY_FP32, H=2, varlen_seqs=len(lens)), TOL_F32_FRO, None
    x = inputs.make_prefill(w, device=DEV, lengths=lens)
    cu_ck = cu_ckpt_for(x, every)
    o, s, ck = kda.kda_chunk_fwd_ckpt(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], every,
                                      initial_state=x["initial_state"], cu_seqlens=x["cu_seqlens"],
                                      cu_ckpt=cu_ck, kernel=kernel, validate=True)
    torch.cuda.synchronize()
    o_ref, s_ref, ck_ref, cu_ref = oracle_ckpt(x, every)
    assert list(cu_ck.cpu().numpy()) == list(cu_ref)
    assert ck.shape[0] == len(ck_ref) == 2 + 0 + 1 + 5 + 0 + 4
    assert_close(to_np(ck), ck_ref, fro, maxn, what="checkpoints")
    assert_close(to_np(o), o_ref, fro, maxn, what="o")
    assert_close(to_np(s), s_ref, fro, maxn, what="S")


def test_ckpt_batch_and_segments(kda):
    """A B x T batch (slots n*(T//every) + j, no cu_ckpt) on the tensor-core
    kernel, unsplit and split into segments (the checkpoints come from the
    rerun of every segment)."""
    every = 256
    w = inputs.scaled(inputs.PREFILL_B4_T8K, B=2, T=1600, H=2)
    x = inputs.make_prefill(w, device=DEV)
    o_ref, s_ref, ck_ref, _ = oracle_ckpt(x, every)
    for segments in (1, 3):
        o, s, ck = kda.kda_chunk_fwd_ckpt(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], every,
                                          initial_state=x["initial_state"], kernel="tc", segments=segments,
                                          B=2)
        torch.cuda.synchronize()
        assert ck.shape[0] == 2 * (1600 // every)
        assert_close(to_np(ck), ck_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what=f"checkpoints, segments={segments}")
        assert_close(to_np(o), o_ref, TOL_BF16_FRO, TOL_BF16_MAXN, what="o")


def test_resume_from_a_checkpoint(kda):
    """Prefix-cache reuse end to end: the state stored after 512 tokens, fed
    back as the initial state of the remaining tokens, gives the outputs and
    final state of the full run (up to bf16 rounding)."""
    every, cut = 256, 512
    w = inputs.scaled(inputs.PREFILL_B4_T8K, B=1, T=1000, H=4)
    x = inputs.make_prefill(w, device=DEV)
    o, s, ck = kda.kda_chunk_fwd_ckpt(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], every,
                                      initial_state=x["initial_state"], kernel="tc", B=1)
    j = cut // every
    o2, s2 = kda.kda_chunk_fwd(x["q"][cut:], x["k"][cut:], x["v"][cut:], x["log_alpha"][cut:],
                               x["beta"][cut:], ck[j - 1:j].contiguous(), None, kernel="tc", B=1)
    torch.cuda.synchronize()
    assert_close(to_np(o2), to_np(o[cut:]), TOL_BF16_FRO, TOL_BF16_MAXN, what="resumed o")
    assert_close(to_np(s2), to_np(s), TOL_BF16_FRO, TOL_BF16_MAXN, what="resumed S")


def test_ckpt_validate_rejects_wrong_slot_counts(kda):
    lens = np.array([300, 200])
    x = inputs.make_prefill(inputs.scaled(inputs.VARLEN_64, H=2), device=DEV, lengths=lens)
    bad = torch.tensor([0, 3, 4], dtype=torch.int32, device=DEV)  # 300 // 128 is 2, not 3
    with pytest.raises(kda.KdaError):
        kda.kda_chunk_fwd_ckpt(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], 128,
                               cu_seqlens=x["cu_seqlens"], cu_ckpt=bad, kernel="tc", validate=True)
