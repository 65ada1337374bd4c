"""Shared test helpers: error metrics and oracle calls on host copies."""
import numpy as np
import torch

import oracle
from hybrid_linear_attention_chunk_gb300 import inputs

# Tolerances for results checked against the fp64 oracle.  fp32 inputs and
# arithmetic: relative Frobenius 1e-4.  bf16 inputs with bf16 tensor-core
# operands and fp32 state: relative Frobenius 2e-2 and max-normalised 5e-2.
TOL_F32_FRO = 1e-4
TOL_BF16_FRO = 2e-2
TOL_BF16_MAXN = 5e-2


def rel_fro(x, y):
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    return float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300))


def max_norm(x, y):
    """max|x - y| / max|y| over the tensor."""
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    return float(np.max(np.abs(x - y)) / max(np.max(np.abs(y)), 1e-300))


def to_np(t):
    return t.detach().float().cpu().numpy()


def oracle_prefill(x, chains=None, nthreads=None):
    h = {n: inputs.host_f32(x[n]) for n in ("q", "k", "v", "log_alpha", "beta", "initial_state")}
    cu = x["cu_seqlens"].cpu().numpy().astype(np.int64)
    return oracle.recurrent(h["q"], h["k"], h["v"], h["log_alpha"], h["beta"], h["initial_state"], cu,
                            chains=chains, nthreads=nthreads)


def assert_close(got, want, fro_tol, maxn_tol=None, what=""):
    e = rel_fro(got, want)
    assert e <= fro_tol, f"{what}: rel-Frobenius {e:.3e} > {fro_tol:.1e}"
    if maxn_tol is not None:
        m = max_norm(got, want)
        assert m <= maxn_tol, f"{what}: max-normalised {m:.3e} > {maxn_tol:.1e}"
    return e


def oracle_heads_by_columns(x, heads, width=16, workers=None):
    """The fp64 oracle on some heads of a packed batch, each head run as
    dv / width independent chains of `width` state columns.

    Under S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
    and o_t = S_t^T q_t, column j of S and output channel j never read another
    column (column j is written by entry j of v alone), so each group of
    columns is the same recurrence with the same q, k, alpha and beta and its
    own slice of v and of the initial state.  Splitting a head this way lets
    the oracle use several host cores on one long sequence; the split itself is
    pinned on the CPU against the unsplit oracle.  Returns (o [T_total,
    len(heads), dv], S [N, len(heads), dk, dv]) in fp64.
    """
    import concurrent.futures as cf
    heads = list(heads)
    dev = x["q"].device
    hs = torch.as_tensor(heads, device=dev)
    cu = x["cu_seqlens"].cpu().numpy().astype(np.int64)
    N = len(cu) - 1
    pick = lambda t: None if t is None else inputs.host_f32(t.index_select(1, hs).contiguous())
    q, k, v, g, s0 = (pick(x[n]) for n in ("q", "k", "v", "log_alpha", "initial_state"))
    beta = pick(x["beta"])
    T, nh, dk = q.shape
    dv = v.shape[2]
    per_head = [tuple(np.ascontiguousarray(a[:, i:i + 1]) for a in (q, k, g, beta)) for i in range(nh)]
    o = np.empty((T, nh, dv))
    S = np.empty((N, nh, dk, dv))

    def run(job):
        i, c0 = job
        sl = slice(c0, min(c0 + width, dv))
        qh, kh, gh, bh = per_head[i]
        vs = np.ascontiguousarray(v[:, i:i + 1, sl])
        ss0 = None if s0 is None else np.ascontiguousarray(s0[:, i:i + 1, :, sl])
        oo, sf = oracle.recurrent(qh, kh, vs, gh, bh, ss0, cu, nthreads=1)
        o[:, i, sl] = oo[:, 0]
        S[:, i, :, sl] = sf[:, 0]

    jobs = [(i, c0) for i in range(nh) for c0 in range(0, dv, width)]
    with cf.ThreadPoolExecutor(workers or oracle.default_threads()) as ex:
        list(ex.map(run, jobs))
    return o, S
