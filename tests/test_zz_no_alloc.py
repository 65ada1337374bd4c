"""The allocation-free prefill entry point, kda_chunk_fwd_noalloc.

It exists for callers that cannot allocate device memory themselves (their
allocator owns the whole GPU, or an allocation on their path could stall or
fail).  It must give the same results as kda_chunk_fwd while taking the
long-sequence workspace from the library's static array.  This file sorts
last so that a run stopping at the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from _helpers import TOL_BF16_FRO, TOL_BF16_MAXN, assert_close, to_np
from hybrid_linear_attention_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _pool_watch():
    """Reset and read the high-water mark of memory in use from the current
    device's memory pool, the pool that stream-ordered allocations
    (cudaMallocAsync) draw from; torch's caching allocator does not use it."""
    rt = None
    for name in ("libcudart.so.13", "libcudart.so", "/usr/local/cuda/lib64/libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            continue
    if rt is None:
        pytest.fail("libcudart not found")
    used_mem_high = 8  # cudaMemPoolAttrUsedMemHigh
    pool = ctypes.c_void_p()
    assert rt.cudaDeviceGetMemPool(ctypes.byref(pool), torch.cuda.current_device()) == 0

    def reset():
        zero = ctypes.c_uint64(0)
        assert rt.cudaMemPoolSetAttribute(pool, used_mem_high, ctypes.byref(zero)) == 0

    def high():
        v = ctypes.c_uint64(0)
        assert rt.cudaMemPoolGetAttribute(pool, used_mem_high, ctypes.byref(v)) == 0
        return v.value

    return reset, high


def _split_inputs(T, H, seed):
    w = inputs.scaled(inputs.LONG_T1M, B=1, T=T, H=H)
    return inputs.make_prefill(w, device=DEV, seed=seed)


def test_noalloc_matches_kda_chunk_fwd_on_two_calls_in_a_row(kda):
    """Two calls in a row, each on a sequence the planner splits (so the
    static scratch is used and reused), against kda_chunk_fwd."""
    for call, (T, H, seed) in enumerate([(6000, 2, 11), (9000, 3, 12)]):
        x = _split_inputs(T, H, seed)
        d = kda.chunk_desc(x["q"], x["v"], gate_dtype=0, segments=4, B=1)
        need = kda.kda_chunk_fwd_workspace_size(d)
        assert 0 < need <= (32 << 20)
        reset, high = _pool_watch()
        torch.cuda.synchronize()
        reset()
        o_ref, s_ref = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                         x["initial_state"], None, B=1, segments=4)
        o = torch.empty_like(o_ref)
        s = torch.empty_like(s_ref)
        torch.cuda.synchronize()
        # the watch sees the workspace kda_chunk_fwd takes from the pool ...
        assert high() >= need
        reset()
        base = high()  # what the pool still had in use at the reset (normally 0)
        kda.kda_chunk_fwd_noalloc(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["initial_state"],
                                  None, o, s, B=1, segments=4)
        torch.cuda.synchronize()
        # ... and nothing from the allocation-free call
        assert high() == base, "kda_chunk_fwd_noalloc took memory from the stream-ordered pool"
        assert_close(to_np(o), to_np(o_ref), TOL_BF16_FRO, TOL_BF16_MAXN, what=f"o call {call}")
        assert_close(to_np(s), to_np(s_ref), TOL_BF16_FRO, TOL_BF16_MAXN, what=f"S call {call}")


def test_noalloc_unsplit_call_matches(kda):
    """Without a split no scratch is needed; the results equal kda_chunk_fwd's."""
    w = inputs.scaled(inputs.VARLEN_64, H=2)
    x = inputs.make_prefill(w, device=DEV, lengths=np.array([300, 77]))
    o_ref, s_ref = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["initial_state"],
                                     x["cu_seqlens"])
    o, s = kda.kda_chunk_fwd_noalloc(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["initial_state"],
                                     x["cu_seqlens"])
    torch.cuda.synchronize()
    assert_close(to_np(o), to_np(o_ref), TOL_BF16_FRO, TOL_BF16_MAXN, what="o")
    assert_close(to_np(s), to_np(s_ref), TOL_BF16_FRO, TOL_BF16_MAXN, what="S")


def test_noalloc_rejects_plans_beyond_the_static_scratch(kda):
    """Two sequences of 2^20 tokens and 16 heads cut into 16 segments each
    need 86 MiB of scratch, more than the 32 MiB array: the call is refused
    before any launch."""
    lib = kda.load()
    d = kda.KdaChunkDesc()
    d.B, d.T, d.H, d.dk, d.dv, d.chunk = 2, 1 << 20, 16, 128, 128, 64
    d.num_seqs, d.qkv_dtype, d.out_dtype, d.gate_dtype, d.validate, d.kernel, d.segments = 0, 1, 1, 0, 0, 0, 16
    assert kda.kda_chunk_fwd_workspace_size(d) > (32 << 20)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    st = lib.kda_chunk_fwd_noalloc(ctypes.byref(d), fake, fake, fake, fake, fake, None, None, fake, None, None)
    assert st == -9
    d.validate = 1
    assert lib.kda_chunk_fwd_noalloc(ctypes.byref(d), fake, fake, fake, fake, fake, None, None, fake, None,
                                     None) == -7
