"""Pins for the oracle's backward (``oracle.backward``).

Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
(liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.  [K3-notes §2.2]
gives the recurrence S_t = (I - b k k^T) Diag(a) S_{t-1} + b k v^T, o_t = S_t^T q_t
and says the chunk form serves training, without printing a backward.  The
gradients are those of L = sum_t <dO_t, o_t> + <dS_T, S_T>.

The main pin is the derivative itself: every gradient entry of a small packed
problem is compared with a Richardson-extrapolated central difference of the
forward oracle.  The inputs are multiples of 2^-6 below 8 in magnitude, so the
perturbed inputs (steps 2^-10 and 2^-11) are exact in the float32 the oracle
takes, and the forward runs in fp64.  Closed forms and planted mistakes
complete it.
"""
import numpy as np
import pytest

import oracle


def f32(x):
    return np.asarray(x, dtype=np.float32)


def grid(rng, shape, lo, hi):
    """Uniform values on the 2^-6 grid in [lo, hi]."""
    return f32(np.round(rng.uniform(lo, hi, shape) * 64.0) / 64.0)


def small_problem(seed=5, dk=3, dv=2, H=2, lens=(4, 0, 3)):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, N = int(cu[-1]), len(lens)
    q, k, v = grid(rng, (T, H, dk), -1, 1), grid(rng, (T, H, dk), -1, 1), grid(rng, (T, H, dv), -1, 1)
    g = grid(rng, (T, H, dk), -1.5, -0.05)
    beta = grid(rng, (T, H), 0.1, 0.95)
    s0 = rng.standard_normal((N, H, dk, dv)) * 0.5
    dO = grid(rng, (T, H, dv), -1, 1)
    dST = grid(rng, (N, H, dk, dv), -1, 1)
    return dict(q=q, k=k, v=v, g=g, beta=beta, s0=s0, dO=dO, dST=dST, cu=cu)


def loss(p, **over):
    a = {**p, **over}
    o, S = oracle.recurrent(a["q"], a["k"], a["v"], a["g"], a["beta"], a["s0"], a["cu"], nthreads=1)
    return float(np.sum(o * a["dO"].astype(np.float64)) + np.sum(S * a["dST"].astype(np.float64)))


def fd_grad(p, name):
    """Richardson-extrapolated central differences of `loss` for every entry of input `name`."""
    x = p[name]
    out = np.zeros(x.shape)
    for idx in np.ndindex(*x.shape):
        d = []
        for h in (2.0 ** -10, 2.0 ** -11):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            d.append((loss(p, **{name: xp}) - loss(p, **{name: xm})) / (2 * h))
        out[idx] = (4 * d[1] - d[0]) / 3
    return out


def grads(p, mutation=0):
    return oracle.backward(p["q"], p["k"], p["v"], p["g"], p["beta"], p["dO"], initial_state=p["s0"],
                           d_final_state=p["dST"], cu_seqlens=p["cu"], nthreads=1, mutation=mutation)


NAMES = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "s0": "ds0"}


def test_every_gradient_entry_matches_finite_differences():
    p = small_problem()
    gr = grads(p)
    for name, gname in NAMES.items():
        fd = fd_grad(p, name)
        scale = max(np.max(np.abs(fd)), 1e-12)
        err = np.max(np.abs(gr[gname] - fd)) / scale
        assert err < 1e-8, f"{gname}: max error {err:.2e} against finite differences"


@pytest.mark.parametrize("mname", sorted(oracle.BWD_MUTATIONS))
def test_planted_backward_mistakes_are_caught(mname):
    p = small_problem()
    gr = grads(p, mutation=oracle.BWD_MUTATIONS[mname])
    worst = 0.0
    for name, gname in NAMES.items():
        fd = fd_grad(p, name)
        worst = max(worst, np.max(np.abs(gr[gname] - fd)) / max(np.max(np.abs(fd)), 1e-12))
    assert worst > 1e-3, f"the finite-difference pin does not catch {mname}"


def test_identity_steps_pass_gradients_through():
    """alpha = 1 and beta = 0 leave the state untouched: S_T = S_0, o_t = S_0^T q_t.
    So dS_0 = dS_T + sum_t q_t dO_t^T, dq_t = S_0 dO_t, and k, v, beta get no
    gradient from the write (dv = 0) while dbeta_t = (dS^T k_t) . (v_t - S_0^T k_t)
    with dS the state gradient after token t."""
    rng = np.random.default_rng(2)
    T, H, dk, dv = 5, 1, 4, 3
    q, k, v = (f32(rng.standard_normal((T, H, d))) for d in (dk, dk, dv))
    g, beta = np.zeros((T, H, dk), np.float32), np.zeros((T, H), np.float32)
    s0 = rng.standard_normal((1, H, dk, dv))
    dO = f32(rng.standard_normal((T, H, dv)))
    dST = f32(rng.standard_normal((1, H, dk, dv)))
    gr = oracle.backward(q, k, v, g, beta, dO, initial_state=s0, d_final_state=dST)
    q, k, v, dO, dST = (x.astype(np.float64) for x in (q, k, v, dO, dST))
    S0 = s0[0, 0]
    dS_after = [dST[0, 0].astype(np.float64) + sum(np.outer(q[s, 0], dO[s, 0]) for s in range(t, T))
                for t in range(T)]
    assert np.allclose(gr["ds0"][0, 0], dS_after[0], rtol=1e-12, atol=1e-12)
    for t in range(T):
        assert np.allclose(gr["dq"][t, 0], S0 @ dO[t, 0], rtol=1e-12, atol=1e-12)
        assert np.allclose(gr["dv"][t, 0], 0.0)
        want_db = (dS_after[t].T @ k[t, 0]) @ (v[t, 0] - S0.T @ k[t, 0])
        assert np.isclose(gr["dbeta"][t, 0], want_db, rtol=1e-12, atol=1e-12)
        # dalpha_i = sum_j dS_ij S0_ij with dS after token t, times alpha = 1
        assert np.allclose(gr["dg"][t, 0], np.sum(dS_after[t] * S0, axis=1), rtol=1e-12, atol=1e-12)


def test_gradient_is_linear_in_the_upstream_gradients():
    p = small_problem(seed=9)
    g1 = grads(p)
    p2 = dict(p, dO=f32(2.0 * p["dO"]), dST=f32(2.0 * p["dST"]))
    g2 = grads(p2)
    for name in g1:
        assert np.allclose(g2[name], 2.0 * g1[name], rtol=1e-12, atol=1e-14)
