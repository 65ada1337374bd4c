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
