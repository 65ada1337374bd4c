"""KDA oracle: plain fp64 CPU reference of the Kimi Delta Attention recurrence.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library in
``hybrid_linear_attention_chunk_gb300`` never imports, links or calls it, and the
two share no code: the C source here is compiled on its own with gcc.

Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
(liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.

Functions (all fp64 inside; inputs are float32 arrays holding the exact values
the GPU receives, so a bf16 input is passed as its exact float32 upcast):

* ``recurrent``     - [K3-notes §2.2, KDA state recurrence], token by token.
* ``chunked``       - [K3-notes §2.2, chunkwise form] with the U, W and carry
                      formulas that the page leaves out (derivation in the C file).
* ``decode_step``   - one token of the recurrence per sequence, state in place.
* ``affine_pair``   - [K3-notes §2.5, context-parallel affine pair] (M, S~).
* ``backward``      - gradients of <dO, o~> + <dS_T, S_T> with respect to every
                      input, by reverse-mode differentiation of the token
                      recurrence (the page names training but prints no backward).
* ``layer``, ``layer_decode_step`` - the recurrence inside the KDA layer's gates
                      ([K3-notes §2.2, Eq. 5 and the KDA output equation]): the
                      log-decay g_min Sigmoid(exp(A_h) z) from decay logits z, and
                      the output Sigmoid(gate) o RMSNorm(o~) per token and head.

Pins that tie these functions to the pages and to mathematics other than
themselves live in ``tests/test_oracle_pins.py``; every function here is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

MUTATIONS = {
    "no_decay": 1,
    "sign_erase": 2,
    "undecayed_predict": 3,
    "read_transposed": 4,
    "read_before_write": 5,
    "beta_only_on_write": 6,
    "decay_by_column": 7,
    "beta_squared": 8,
}

# Planted mistakes in the backward (``backward`` only).
BWD_MUTATIONS = {
    "bwd_ds_undecayed": 16,
    "bwd_dk_no_predict": 17,
    "bwd_dg_from_ds": 18,
}

# Planted mistakes in the layer gates (``layer`` only).
GATE_MUTATIONS = {
    "gate_neg_logit": 9,
    "gate_no_exp": 10,
    "gate_head0": 11,
    "norm_sum": 12,
    "norm_eps_outside": 13,
    "ogate_neg": 14,
    "norm_w_reversed": 15,
}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, no CUDA).  Returns the .so path."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    I = ctypes.c_int
    L = ctypes.c_int64
    lib.oracle_kda_recurrent.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, P, P, I, I, I]
    lib.oracle_kda_recurrent.restype = I
    lib.oracle_kda_chunked.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, P, P, I, I, I, I]
    lib.oracle_kda_chunked.restype = I
    lib.oracle_kda_decode_step.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, I, I]
    lib.oracle_kda_decode_step.restype = I
    lib.oracle_kda_affine_pair.argtypes = [I, I, I, I, L, L, P, P, P, P, P, P]
    lib.oracle_kda_affine_pair.restype = I
    D = ctypes.c_double
    lib.oracle_kda_layer.argtypes = [I, I, I, I, P, P, P, P, P, P, D, P, P, P, D, P, P, P, I, I]
    lib.oracle_kda_layer.restype = I
    lib.oracle_kda_layer_decode_step.argtypes = [I, I, I, I, P, P, P, P, P, D, P, P, P, D, P, P, I]
    lib.oracle_kda_layer_decode_step.restype = I
    lib.oracle_kda_backward.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, I, I]
    lib.oracle_kda_backward.restype = I
    lib.oracle_kda_recurrent_ckpt.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, P, I, P, P, I]
    lib.oracle_kda_recurrent_ckpt.restype = I
    _lib = lib
    return lib


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _prep(q, k, v, g, beta, cu_seqlens):
    q, k, v, g = (np.asarray(x) for x in (q, k, v, g))
    beta = np.asarray(beta)
    if q.ndim != 3:
        raise ValueError("q must be [T_total, H, dk]")
    T, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is None:
        cu_seqlens = np.array([0, T], dtype=np.int64)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    N = len(cu) - 1
    if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0, end at T_total and not decrease")
    arrs = [_f32(x) for x in (q, k, v, g, beta)]
    return T, H, dk, dv, N, cu, arrs


def _chains(chains):
    if chains is None:
        return None, None, 0
    c = np.ascontiguousarray(np.asarray(chains, dtype=np.int32))
    return c, c.ctypes.data_as(ctypes.c_void_p), len(c)


def recurrent(q, k, v, g, beta, initial_state=None, cu_seqlens=None, chains=None,
              nthreads=None, mutation: int = 0, want_o: bool = True):
    """Token-by-token KDA recurrence in fp64.

    q, k, g: [T_total, H, dk]; v: [T_total, H, dv]; beta: [T_total, H];
    initial_state: [N, H, dk, dv] or None (zeros); cu_seqlens: [N+1] or None
    (one sequence).  chains: optional list of n*H+h to compute (others: o rows
    stay NaN and states stay NaN).  Returns (o [T_total,H,dv], S [N,H,dk,dv]).
    """
    lib = _load()
    T, H, dk, dv, N, cu, arrs = _prep(q, k, v, g, beta, cu_seqlens)
    s0 = None if initial_state is None else _f64(initial_state)[0]
    o = np.full((T, H, dv), np.nan) if want_o else None
    sf = np.full((N, H, dk, dv), np.nan)
    c, cp, nc = _chains(chains)
    st = lib.oracle_kda_recurrent(N, H, dk, dv, cu.ctypes.data_as(ctypes.c_void_p),
                                  *[a[1] for a in arrs], _ptr(s0), _ptr(o), _ptr(sf), cp, nc,
                                  nthreads or default_threads(), int(mutation))
    if st != 0:
        raise RuntimeError(f"oracle_kda_recurrent failed with {st}")
    return o, sf


def recurrent_ckpt(q, k, v, g, beta, every, initial_state=None, cu_seqlens=None, nthreads=None,
                   want_o: bool = True):
    """The fp64 token recurrence that also records each sequence's state after
    every `every` tokens ([K3-notes §2.5, Fig. 12]: the state at a prefix's end
    is what a request sharing that prefix resumes from).

    Returns (o, S_final, ckpt [slots, H, dk, dv], cu_ckpt [N+1]) where sequence
    n's j-th checkpoint (after its first j*every tokens) is slot cu_ckpt[n] + j - 1.
    """
    lib = _load()
    T, H, dk, dv, N, cu, arrs = _prep(q, k, v, g, beta, cu_seqlens)
    s0 = None if initial_state is None else _f64(initial_state)[0]
    o = np.full((T, H, dv), np.nan) if want_o else None
    sf = np.full((N, H, dk, dv), np.nan)
    cu_ck = np.zeros(N + 1, dtype=np.int64)
    cu_ck[1:] = np.cumsum(np.diff(cu) // int(every))
    ck = np.full((max(int(cu_ck[-1]), 1), H, dk, dv), np.nan)
    st = lib.oracle_kda_recurrent_ckpt(N, H, dk, dv, cu.ctypes.data_as(ctypes.c_void_p),
                                       *[a[1] for a in arrs], _ptr(s0), _ptr(o), _ptr(sf), int(every),
                                       cu_ck.ctypes.data_as(ctypes.c_void_p), _ptr(ck),
                                       nthreads or default_threads())
    if st != 0:
        raise RuntimeError(f"oracle_kda_recurrent_ckpt failed with {st}")
    return o, sf, ck[:int(cu_ck[-1])], cu_ck


def chunked(q, k, v, g, beta, initial_state=None, cu_seqlens=None, chunk=64, subtile_ref=False,
            chains=None, nthreads=None):
    """fp64 chunkwise form (same arguments and returns as ``recurrent``)."""
    lib = _load()
    T, H, dk, dv, N, cu, arrs = _prep(q, k, v, g, beta, cu_seqlens)
    s0 = None if initial_state is None else _f64(initial_state)[0]
    o = np.full((T, H, dv), np.nan)
    sf = np.full((N, H, dk, dv), np.nan)
    c, cp, nc = _chains(chains)
    st = lib.oracle_kda_chunked(N, H, dk, dv, cu.ctypes.data_as(ctypes.c_void_p),
                                *[a[1] for a in arrs], _ptr(s0), _ptr(o), _ptr(sf), cp, nc,
                                nthreads or default_threads(), int(chunk), int(bool(subtile_ref)))
    if st != 0:
        raise RuntimeError(f"oracle_kda_chunked failed with {st}")
    return o, sf


def decode_step(q, k, v, g, beta, state, chains=None, nthreads=None):
    """One decode step: q,k,g [N,H,dk], v [N,H,dv], beta [N,H], state [N,H,dk,dv].

    Returns (o [N,H,dv], new_state).  The input state array is not modified.
    """
    lib = _load()
    q, k, v, g = (np.asarray(x) for x in (q, k, v, g))
    N, H, dk = q.shape
    dv = v.shape[2]
    arrs = [_f32(x) for x in (q, k, v, g, beta)]
    S = np.array(state, dtype=np.float64, copy=True, order="C")
    o = np.full((N, H, dv), np.nan)
    c, cp, nc = _chains(chains)
    st = lib.oracle_kda_decode_step(N, H, dk, dv, *[a[1] for a in arrs], _ptr(S), _ptr(o), cp, nc,
                                    nthreads or default_threads())
    if st != 0:
        raise RuntimeError(f"oracle_kda_decode_step failed with {st}")
    return o, S


def affine_pair(k, v, g, beta, h, t0, t1):
    """(M, S~) of tokens [t0, t1) of head h: S_out = S~ + M S_in."""
    lib = _load()
    k, v, g = (np.asarray(x) for x in (k, v, g))
    T, H, dk = k.shape
    dv = v.shape[2]
    arrs = [_f32(x) for x in (k, v, g, beta)]
    M = np.zeros((dk, dk))
    St = np.zeros((dk, dv))
    st = lib.oracle_kda_affine_pair(H, dk, dv, int(h), int(t0), int(t1), *[a[1] for a in arrs],
                                    _ptr(M), _ptr(St))
    if st != 0:
        raise RuntimeError(f"oracle_kda_affine_pair failed with {st}")
    return M, St


def layer(q, k, v, z, beta, A_log, g_min=-5.0, out_gate=None, norm_weight=None, norm_eps=1e-6,
          initial_state=None, cu_seqlens=None, nthreads=None, mutation: int = 0):
    """The KDA recurrence inside the layer's gates, in fp64.

    z: [T_total, H, dk] decay logits, A_log: [H]; the log-decay is
    g_min * Sigmoid(exp(A_log[h]) * z) ([K3-notes §2.2, Eq. 5]).  out_gate:
    [T_total, H, dv] output gate logits (W_g x) or None; when given, each output
    row becomes Sigmoid(out_gate) * o / sqrt(mean(o^2) + norm_eps) * norm_weight
    ([K3-notes §2.2, KDA output]); norm_weight [dv] or None (ones).  Other
    arguments and the returns (o, S_final) as ``recurrent``.
    """
    lib = _load()
    T, H, dk, dv, N, cu, arrs = _prep(q, k, v, z, beta, cu_seqlens)
    A, pA = _f32(np.asarray(A_log).reshape(-1))
    if A.shape[0] != H:
        raise ValueError("A_log must have H entries")
    og = None if out_gate is None else _f32(out_gate)
    w = None if norm_weight is None else _f32(np.asarray(norm_weight).reshape(-1))
    s0 = None if initial_state is None else _f64(initial_state)[0]
    o = np.full((T, H, dv), np.nan)
    sf = np.full((N, H, dk, dv), np.nan)
    st = lib.oracle_kda_layer(N, H, dk, dv, cu.ctypes.data_as(ctypes.c_void_p), arrs[0][1], arrs[1][1],
                              arrs[2][1], arrs[3][1], pA, float(g_min), arrs[4][1],
                              None if og is None else og[1], None if w is None else w[1], float(norm_eps),
                              _ptr(s0), _ptr(o), _ptr(sf), nthreads or default_threads(), int(mutation))
    if st != 0:
        raise RuntimeError(f"oracle_kda_layer failed with {st}")
    return o, sf


def layer_decode_step(q, k, v, z, beta, state, A_log, g_min=-5.0, out_gate=None, norm_weight=None,
                      norm_eps=1e-6, nthreads=None):
    """One decode step of ``layer``: q, k, z [N,H,dk], v [N,H,dv], beta [N,H],
    out_gate [N,H,dv] or None, state [N,H,dk,dv].  Returns (o, new_state); the
    input state is not modified."""
    lib = _load()
    q, k, v, z = (np.asarray(x) for x in (q, k, v, z))
    N, H, dk = q.shape
    dv = v.shape[2]
    arrs = [_f32(x) for x in (q, k, v, z, beta)]
    A, pA = _f32(np.asarray(A_log).reshape(-1))
    og = None if out_gate is None else _f32(out_gate)
    w = None if norm_weight is None else _f32(np.asarray(norm_weight).reshape(-1))
    S = np.array(state, dtype=np.float64, copy=True, order="C")
    o = np.full((N, H, dv), np.nan)
    st = lib.oracle_kda_layer_decode_step(N, H, dk, dv, arrs[0][1], arrs[1][1], arrs[2][1], arrs[3][1], pA,
                                          float(g_min), arrs[4][1], None if og is None else og[1],
                                          None if w is None else w[1], float(norm_eps), _ptr(S), _ptr(o),
                                          nthreads or default_threads())
    if st != 0:
        raise RuntimeError(f"oracle_kda_layer_decode_step failed with {st}")
    return o, S


def backward(q, k, v, g, beta, d_out, initial_state=None, d_final_state=None, cu_seqlens=None,
             nthreads=None, mutation: int = 0):
    """fp64 gradients of L = sum_t <d_out_t, o~_t> + <d_final_state, S_T>.

    Arguments as ``recurrent`` plus d_out [T_total, H, dv] and d_final_state
    [N, H, dk, dv] (None: 0), both float32 like the other inputs.  Returns a
    dict with dq, dk [T_total,H,dk], dv [T_total,H,dv], dg (log-decay)
    [T_total,H,dk], dbeta [T_total,H] and ds0 [N,H,dk,dv].
    """
    lib = _load()
    T, H, dk, dv, N, cu, arrs = _prep(q, k, v, g, beta, cu_seqlens)
    s0 = None if initial_state is None else _f64(initial_state)[0]
    dO = _f32(d_out)
    dST = None if d_final_state is None else _f32(d_final_state)
    out = dict(dq=np.zeros((T, H, dk)), dk=np.zeros((T, H, dk)), dv=np.zeros((T, H, dv)),
               dg=np.zeros((T, H, dk)), dbeta=np.zeros((T, H)), ds0=np.zeros((N, H, dk, dv)))
    st = lib.oracle_kda_backward(N, H, dk, dv, cu.ctypes.data_as(ctypes.c_void_p), *[a[1] for a in arrs],
                                 _ptr(s0), dO[1], None if dST is None else dST[1], _ptr(out["dq"]),
                                 _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]), _ptr(out["dbeta"]),
                                 _ptr(out["ds0"]), nthreads or default_threads(), int(mutation))
    if st != 0:
        raise RuntimeError(f"oracle_kda_backward failed with {st}")
    return out
