"""ctypes binding of libkda.so (include/kda.h).  Argument marshalling only.

Every step of the computation runs in the library's CUDA kernels.  PyTorch
supplies device memory and the current stream.  There is no fallback: if
libkda.so is missing or cannot load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_F32, KDA_BF16 = 0, 1
KERNELS = {"auto": 0, "simt": 1, "tc": 2}
STATUS = {
    0: "KDA_OK", -1: "KDA_ERR_NULL", -2: "KDA_ERR_SHAPE", -3: "KDA_ERR_DTYPE",
    -4: "KDA_ERR_ALIGN", -5: "KDA_ERR_RANGE", -6: "KDA_ERR_CUDA", -7: "KDA_ERR_UNSUPPORTED",
    -8: "KDA_ERR_ALIAS", -9: "KDA_ERR_SCRATCH_LIMIT",
}


class KdaChunkDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("chunk", ctypes.c_int),
                ("num_seqs", ctypes.c_int), ("qkv_dtype", ctypes.c_int),
                ("out_dtype", ctypes.c_int), ("gate_dtype", ctypes.c_int),
                ("validate", ctypes.c_int), ("kernel", ctypes.c_int), ("segments", ctypes.c_int)]


class KdaDecodeDesc(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int), ("H", ctypes.c_int), ("dk", ctypes.c_int),
                ("dv", ctypes.c_int), ("qkv_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("gate_dtype", ctypes.c_int), ("validate", ctypes.c_int)]


class KdaLayerGates(ctypes.Structure):
    _fields_ = [("A_log", ctypes.c_void_p), ("g_min", ctypes.c_float), ("out_gate", ctypes.c_void_p),
                ("norm_weight", ctypes.c_void_p), ("norm_eps", ctypes.c_float)]


class KdaError(RuntimeError):
    def __init__(self, status: int, fn: str, detail: str = ""):
        self.status = status
        name = STATUS.get(status, str(status))
        super().__init__(f"{fn} returned {name}" + (f": {detail}" if detail else ""))


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libkda.so (raises if it is absent: there is no CPU path)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkda.so is not built ({LIB_PATH}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        lib.kda_chunk_fwd.argtypes = [ctypes.POINTER(KdaChunkDesc), P, P, P, P, P, P, P, P, P, P]
        lib.kda_chunk_fwd.restype = ctypes.c_int
        lib.kda_chunk_fwd_ex.argtypes = [ctypes.POINTER(KdaChunkDesc), P, P, P, P, P, P, P, P, P,
                                         P, ctypes.c_size_t, P]
        lib.kda_chunk_fwd_ex.restype = ctypes.c_int
        lib.kda_chunk_fwd_workspace_size.argtypes = [ctypes.POINTER(KdaChunkDesc),
                                                     ctypes.POINTER(ctypes.c_size_t)]
        lib.kda_chunk_fwd_workspace_size.restype = ctypes.c_int
        lib.kda_chunk_fwd_noalloc.argtypes = [ctypes.POINTER(KdaChunkDesc), P, P, P, P, P, P, P, P, P, P]
        lib.kda_chunk_fwd_noalloc.restype = ctypes.c_int
        lib.kda_chunk_fwd_ckpt.argtypes = [ctypes.POINTER(KdaChunkDesc), P, P, P, P, P, P, P, P, P,
                                           ctypes.c_int, P, P, P, ctypes.c_size_t, P]
        lib.kda_chunk_fwd_ckpt.restype = ctypes.c_int
        lib.kda_decode_step.argtypes = [ctypes.POINTER(KdaDecodeDesc), P, P, P, P, P, P, P, P]
        lib.kda_decode_step.restype = ctypes.c_int
        lib.kda_layer_fwd.argtypes = [ctypes.POINTER(KdaChunkDesc), ctypes.POINTER(KdaLayerGates), P, P, P, P, P,
                                      P, P, P, P, P, ctypes.c_size_t, P]
        lib.kda_layer_fwd.restype = ctypes.c_int
        lib.kda_layer_decode_step.argtypes = [ctypes.POINTER(KdaDecodeDesc), ctypes.POINTER(KdaLayerGates), P, P,
                                              P, P, P, P, P, P]
        lib.kda_layer_decode_step.restype = ctypes.c_int
        lib.kda_chunk_bwd_workspace_size.argtypes = [ctypes.POINTER(KdaChunkDesc), ctypes.POINTER(ctypes.c_size_t)]
        lib.kda_chunk_bwd_workspace_size.restype = ctypes.c_int
        lib.kda_chunk_bwd.argtypes = [ctypes.POINTER(KdaChunkDesc), P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P,
                                      ctypes.c_size_t, P]
        lib.kda_chunk_bwd.restype = ctypes.c_int
        lib.kda_chunk_affine_pair.argtypes = [ctypes.POINTER(KdaChunkDesc), P, P, P, P, P, P, P, P]
        lib.kda_chunk_affine_pair.restype = ctypes.c_int
        lib.kda_affine_compose.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           P, P, P, P]
        lib.kda_affine_compose.restype = ctypes.c_int
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_last_cuda_error.argtypes = []
        lib.kda_last_cuda_error.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, fn: str):
    if status != 0:
        lib = load()
        detail = lib.kda_status_string(status).decode()
        if status == -6:
            detail += " (" + lib.kda_last_cuda_error().decode() + ")"
        raise KdaError(status, fn, detail)


def chunk_desc(q, v, *, chunk=64, cu_seqlens=None, out_dtype=None, gate_dtype=None, validate=False,
               kernel="auto", segments=0, B=None) -> KdaChunkDesc:
    if q.dim() == 4:
        B_, T, H, dk = q.shape
    else:
        T, H, dk = q.shape
        B_ = 1
    if B is not None and q.dim() == 3:
        B_ = B
        T = T // B
    dv = v.shape[-1]
    d = KdaChunkDesc()
    d.B, d.T, d.H, d.dk, d.dv, d.chunk = B_, T, H, dk, dv, chunk
    d.num_seqs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    d.qkv_dtype = _dt(q)
    d.out_dtype = KDA_BF16 if out_dtype == torch.bfloat16 else (
        KDA_F32 if out_dtype == torch.float32 else _dt(q))
    d.gate_dtype = gate_dtype if gate_dtype is not None else KDA_F32
    d.validate = int(bool(validate))
    d.kernel = KERNELS[kernel]
    d.segments = int(segments)
    return d


def kda_chunk_fwd(q, k, v, log_alpha, beta, initial_state=None, cu_seqlens=None, out=None,
                  final_state=None, *, chunk=64, kernel="auto", segments=0, validate=False,
                  out_dtype=None, want_final_state=True, B=None, stream=None, workspace=None):
    """Chunked KDA prefill through the C ABI.

    q, k, log_alpha: [B*T, H, dk] (or [B, T, H, dk]); v: [.., H, dv];
    beta: [B*T, H]; initial_state: [N, H, dk, dv] fp32 or None;
    cu_seqlens: int32 [N+1] on the device or None.  Returns (out, final_state).
    """
    lib = load()
    dev = q.device
    d = chunk_desc(q, v, chunk=chunk, cu_seqlens=cu_seqlens, out_dtype=out_dtype or q.dtype,
                   gate_dtype=_dt(log_alpha), validate=validate, kernel=kernel, segments=segments, B=B)
    if beta.dtype != log_alpha.dtype:
        raise TypeError("log_alpha and beta must share a dtype")
    Nseq = d.num_seqs if cu_seqlens is not None else d.B
    if out is None:
        out = torch.empty(q.shape[:-1] + (d.dv,), dtype=out_dtype or q.dtype, device=dev)
    if final_state is None and want_final_state:
        final_state = torch.empty(Nseq, d.H, d.dk, d.dv, dtype=torch.float32, device=dev)
    args = [ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
            _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state)]
    if workspace is not None:
        st = lib.kda_chunk_fwd_ex(*args, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream_handle(stream, dev))
        _check(st, "kda_chunk_fwd_ex")
    else:
        st = lib.kda_chunk_fwd(*args, _stream_handle(stream, dev))
        _check(st, "kda_chunk_fwd")
    return out, final_state


def kda_chunk_fwd_noalloc(q, k, v, log_alpha, beta, initial_state=None, cu_seqlens=None, out=None,
                          final_state=None, *, chunk=64, kernel="auto", segments=0, out_dtype=None,
                          want_final_state=True, B=None, stream=None):
    """kda_chunk_fwd through the entry point that allocates no device memory:
    the long-sequence workspace comes from the library's static scratch array
    (KDA_STATIC_WORKSPACE_BYTES).  Output tensors are allocated here by torch
    only when not given; pass `out` and `final_state` to allocate nothing."""
    lib = load()
    dev = q.device
    d = chunk_desc(q, v, chunk=chunk, cu_seqlens=cu_seqlens, out_dtype=out_dtype or q.dtype,
                   gate_dtype=_dt(log_alpha), validate=False, kernel=kernel, segments=segments, B=B)
    Nseq = d.num_seqs if cu_seqlens is not None else d.B
    if out is None:
        out = torch.empty(q.shape[:-1] + (d.dv,), dtype=out_dtype or q.dtype, device=dev)
    if final_state is None and want_final_state:
        final_state = torch.empty(Nseq, d.H, d.dk, d.dv, dtype=torch.float32, device=dev)
    st = lib.kda_chunk_fwd_noalloc(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                   _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                   _stream_handle(stream, dev))
    _check(st, "kda_chunk_fwd_noalloc")
    return out, final_state


def kda_chunk_fwd_ckpt(q, k, v, log_alpha, beta, every, initial_state=None, cu_seqlens=None,
                       cu_ckpt=None, out=None, final_state=None, ckpt=None, *, chunk=64, kernel="auto",
                       segments=0, validate=False, out_dtype=None, want_final_state=True, B=None,
                       stream=None, workspace=None):
    """kda_chunk_fwd that also stores the fp32 state after every `every`
    tokens of each sequence (prefix-cache checkpoints).

    cu_ckpt: int32 [N+1] on the device with cu_ckpt[n+1] - cu_ckpt[n] =
    len_n // every (required with cu_seqlens).  When `ckpt` is None it is
    allocated here with cu_ckpt[-1] slots (a device-to-host read) or, for a
    B x T batch, B * (T // every) slots.  Returns (out, final_state, ckpt).
    """
    lib = load()
    dev = q.device
    d = chunk_desc(q, v, chunk=chunk, cu_seqlens=cu_seqlens, out_dtype=out_dtype or q.dtype,
                   gate_dtype=_dt(log_alpha), validate=validate, kernel=kernel, segments=segments, B=B)
    Nseq = d.num_seqs if cu_seqlens is not None else d.B
    if out is None:
        out = torch.empty(q.shape[:-1] + (d.dv,), dtype=out_dtype or q.dtype, device=dev)
    if final_state is None and want_final_state:
        final_state = torch.empty(Nseq, d.H, d.dk, d.dv, dtype=torch.float32, device=dev)
    if ckpt is None:
        slots = int(cu_ckpt[-1].item()) if cu_seqlens is not None else d.B * (d.T // every if every > 0 else 0)
        ckpt = torch.empty(max(slots, 1), d.H, d.dk, d.dv, dtype=torch.float32, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.kda_chunk_fwd_ckpt(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                int(every), _ptr(cu_ckpt), _ptr(ckpt), _ptr(workspace), ws_bytes,
                                _stream_handle(stream, dev))
    _check(st, "kda_chunk_fwd_ckpt")
    return out, final_state, ckpt


def kda_chunk_fwd_workspace_size(desc: KdaChunkDesc) -> int:
    lib = load()
    n = ctypes.c_size_t(0)
    _check(lib.kda_chunk_fwd_workspace_size(ctypes.byref(desc), ctypes.byref(n)),
           "kda_chunk_fwd_workspace_size")
    return n.value


def kda_decode_step(q, k, v, log_alpha, beta, state_inout, out=None, *, validate=False,
                    out_dtype=None, stream=None):
    """One decode step through the C ABI: q,k,log_alpha [N,H,dk], v [N,H,dv],
    beta [N,H], state_inout [N,H,dk,dv] fp32 (updated in place).  Returns out."""
    lib = load()
    N, H, dk = q.shape
    dv = v.shape[-1]
    d = KdaDecodeDesc()
    d.N, d.H, d.dk, d.dv = N, H, dk, dv
    d.qkv_dtype = _dt(q)
    od = out_dtype or q.dtype
    d.out_dtype = _dt(torch.empty(0, dtype=od))
    d.gate_dtype = _dt(log_alpha)
    d.validate = int(bool(validate))
    if out is None:
        out = torch.empty(N, H, dv, dtype=od, device=q.device)
    st = lib.kda_decode_step(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                             _ptr(state_inout), _ptr(out), _stream_handle(stream, q.device))
    _check(st, "kda_decode_step")
    return out


def layer_gates(A_log, g_min=-5.0, out_gate=None, norm_weight=None, norm_eps=1e-6) -> KdaLayerGates:
    """The kda_layer_gates struct for the given device tensors."""
    lg = KdaLayerGates()
    lg.A_log = None if A_log is None else A_log.data_ptr()
    lg.g_min = float(g_min)
    lg.out_gate = None if out_gate is None else _ptr(out_gate).value
    lg.norm_weight = None if norm_weight is None else _ptr(norm_weight).value
    lg.norm_eps = float(norm_eps)
    return lg


def kda_layer_fwd(q, k, v, z, beta, A_log, g_min=-5.0, out_gate=None, norm_weight=None, norm_eps=1e-6,
                  initial_state=None, cu_seqlens=None, out=None, final_state=None, *, chunk=64, kernel="auto",
                  segments=0, validate=False, out_dtype=None, want_final_state=True, B=None, stream=None,
                  workspace=None):
    """KDA prefill inside the layer's gates through the C ABI: the log-decay is
    g_min * sigmoid(exp(A_log[h]) * z) (z: [.., H, dk] decay logits in q's
    dtype; A_log: [H] fp32) and, with out_gate ([.., H, dv], q's dtype), the
    output is sigmoid(out_gate) * RMSNorm(o) with norm_weight [dv] fp32 (None:
    ones) and norm_eps.  beta: fp32 or bf16.  Returns (out, final_state)."""
    lib = load()
    dev = q.device
    if z.dtype != q.dtype:
        raise TypeError("z must have q's dtype")
    if out_gate is not None and out_gate.dtype != q.dtype:
        raise TypeError("out_gate must have q's dtype")
    d = chunk_desc(q, v, chunk=chunk, cu_seqlens=cu_seqlens, out_dtype=out_dtype or q.dtype,
                   gate_dtype=_dt(beta), validate=validate, kernel=kernel, segments=segments, B=B)
    Nseq = d.num_seqs if cu_seqlens is not None else d.B
    if out is None:
        out = torch.empty(q.shape[:-1] + (d.dv,), dtype=out_dtype or q.dtype, device=dev)
    if final_state is None and want_final_state:
        final_state = torch.empty(Nseq, d.H, d.dk, d.dv, dtype=torch.float32, device=dev)
    lg = layer_gates(A_log, g_min, out_gate, norm_weight, norm_eps)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.kda_layer_fwd(ctypes.byref(d), ctypes.byref(lg), _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta),
                           _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                           _ptr(workspace), ws_bytes, _stream_handle(stream, dev))
    _check(st, "kda_layer_fwd")
    return out, final_state


def kda_layer_decode_step(q, k, v, z, beta, state_inout, A_log, g_min=-5.0, out_gate=None, norm_weight=None,
                          norm_eps=1e-6, out=None, *, validate=False, out_dtype=None, stream=None):
    """One decode step inside the layer's gates (see kda_layer_fwd): q, k, z
    [N,H,dk], v and out_gate [N,H,dv], beta [N,H], state_inout [N,H,dk,dv] fp32
    updated in place.  Returns out."""
    lib = load()
    N, H, dk = q.shape
    dv = v.shape[-1]
    d = KdaDecodeDesc()
    d.N, d.H, d.dk, d.dv = N, H, dk, dv
    d.qkv_dtype = _dt(q)
    od = out_dtype or q.dtype
    d.out_dtype = _dt(torch.empty(0, dtype=od))
    d.gate_dtype = _dt(beta)
    d.validate = int(bool(validate))
    if out is None:
        out = torch.empty(N, H, dv, dtype=od, device=q.device)
    lg = layer_gates(A_log, g_min, out_gate, norm_weight, norm_eps)
    st = lib.kda_layer_decode_step(ctypes.byref(d), ctypes.byref(lg), _ptr(q), _ptr(k), _ptr(v), _ptr(z),
                                   _ptr(beta), _ptr(state_inout), _ptr(out), _stream_handle(stream, q.device))
    _check(st, "kda_layer_decode_step")
    return out


def kda_chunk_bwd_workspace_size(desc: KdaChunkDesc) -> int:
    lib = load()
    n = ctypes.c_size_t(0)
    _check(lib.kda_chunk_bwd_workspace_size(ctypes.byref(desc), ctypes.byref(n)), "kda_chunk_bwd_workspace_size")
    return n.value


def kda_chunk_bwd(q, k, v, log_alpha, beta, d_out, initial_state=None, d_final_state=None, cu_seqlens=None,
                  *, chunk=64, validate=False, want_d_initial_state=True, B=None, stream=None, workspace=None,
                  grads=None):
    """Gradients of kda_chunk_fwd through the C ABI for
    L = sum <d_out, out> + <d_final_state, final_state>.

    Arguments as kda_chunk_fwd plus d_out (out's shape and dtype) and
    d_final_state ([N,H,dk,dv] fp32 or None).  Returns a dict of fp32 tensors
    dq, dk, dv, dlog_alpha, dbeta and d_initial_state (None unless wanted).
    `grads` may pass that dict preallocated."""
    lib = load()
    dev = q.device
    d = chunk_desc(q, v, chunk=chunk, cu_seqlens=cu_seqlens, out_dtype=d_out.dtype, gate_dtype=_dt(log_alpha),
                   validate=validate, B=B)
    Nseq = d.num_seqs if cu_seqlens is not None else d.B
    if grads is None:
        f = dict(dtype=torch.float32, device=dev)
        grads = dict(dq=torch.empty(q.shape, **f), dk=torch.empty(k.shape, **f), dv=torch.empty(v.shape, **f),
                     dlog_alpha=torch.empty(log_alpha.shape, **f), dbeta=torch.empty(beta.shape, **f),
                     d_initial_state=(torch.empty(Nseq, d.H, d.dk, d.dv, **f) if want_d_initial_state else None))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.kda_chunk_bwd(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                           _ptr(initial_state), _ptr(cu_seqlens), _ptr(d_out), _ptr(d_final_state),
                           _ptr(grads["dq"]), _ptr(grads["dk"]), _ptr(grads["dv"]), _ptr(grads["dlog_alpha"]),
                           _ptr(grads["dbeta"]), _ptr(grads.get("d_initial_state")), _ptr(workspace), ws_bytes,
                           _stream_handle(stream, dev))
    _check(st, "kda_chunk_bwd")
    return grads


def kda_chunk_affine_pair(q, k, v, log_alpha, beta, cu_seqlens=None, pairs=None, *, B=None, validate=False,
                          stream=None):
    """The affine pair (S~, M) of each sequence of the call: returns pairs
    [2, N, H, dk, dv] fp32 with pairs[0] = S~ and pairs[1] = M."""
    lib = load()
    d = chunk_desc(q, v, cu_seqlens=cu_seqlens, gate_dtype=_dt(log_alpha), validate=validate, B=B)
    Nseq = d.num_seqs if cu_seqlens is not None else d.B
    if pairs is None:
        pairs = torch.empty(2, Nseq, d.H, d.dk, d.dv, dtype=torch.float32, device=q.device)
    st = lib.kda_chunk_affine_pair(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                   _ptr(cu_seqlens), _ptr(pairs), _stream_handle(stream, q.device))
    _check(st, "kda_chunk_affine_pair")
    return pairs


def kda_affine_compose(pairs, initial_state=None, entry_states=None, *, stream=None):
    """Entry states [N, P, H, dk, dv] of P consecutive segments from the pairs
    [2, N, P-1, H, dk, dv] of the first P-1 and the first entry state."""
    lib = load()
    _, N, Pm1, H, dk, dv = pairs.shape
    P = Pm1 + 1
    if entry_states is None:
        entry_states = torch.empty(N, P, H, dk, dv, dtype=torch.float32, device=pairs.device)
    st = lib.kda_affine_compose(N, H, dk, dv, P, _ptr(initial_state), _ptr(pairs) if Pm1 > 0 else None,
                                _ptr(entry_states), _stream_handle(stream, pairs.device))
    _check(st, "kda_affine_compose")
    return entry_states
