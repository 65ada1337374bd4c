"""Pins for the fp64 oracle: checks against facts other than the oracle itself.

Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
(liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.  The recurrence is
[K3-notes §2.2]: S_t = (I - b k k^T) Diag(a) S_{t-1} + b k v^T, o_t = S_t^T q_t.

Each pin is chosen so that a plausible slip in the oracle (a dropped decay, a
flipped sign, a transposed read-out, beta in the wrong place, the decay on the
wrong index, reading before writing) fails at least one of them;
``test_planted_mistakes_are_caught`` plants each slip in the oracle and checks.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle

RTOL = 1e-12


def f32(x):
    return np.asarray(x, dtype=np.float32)


def exact_unit_keys(rng, T, H, d):
    """Keys with four entries of +-1/2 and the rest 0: unit norm exactly in fp32."""
    k = np.zeros((T, H, d), np.float32)
    for t in range(T):
        for h in range(H):
            idx = rng.choice(d, 4, replace=False)
            k[t, h, idx] = rng.choice([-0.5, 0.5], 4)
    return k


def hadamard(n):
    Hm = np.array([[1.0]])
    while Hm.shape[0] < n:
        Hm = np.block([[Hm, Hm], [Hm, -Hm]])
    return Hm


def rand_inputs(rng, T, H, dk, dv, unit_keys=True, g_lo=math.log(0.5), g_hi=-1e-3):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_keys:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = rng.uniform(g_lo, g_hi, (T, H, dk))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    return [f32(x) for x in (q, k, v, g, beta)]


# ---------------------------------------------------------------- pin suite
# Every pin takes the recurrence as a function so that the planted-mistake
# test can run the same pins against a deliberately broken oracle.

def pin_exact_recall(rec):
    """beta = 1, |k| = 1, q = k  =>  o_t = v_t for any state and decay.
    (I - k k^T) k = 0 erases what the decayed state said about k, and the write
    puts back exactly v ([K3-notes §2.2]: 'erase along the current key, then write')."""
    rng = np.random.default_rng(1)
    T, H, d = 9, 2, 6
    q, k, v, g, beta = rand_inputs(rng, T, H, d, d)
    k = exact_unit_keys(rng, T, H, d)
    q = k.copy()
    beta = np.ones_like(beta)
    s0 = rng.standard_normal((1, H, d, d))
    o, _ = rec(q, k, v, g, beta, s0)
    return np.max(np.abs(o - v.astype(np.float64))) <= 1e-12


def pin_identity(rec):
    """alpha = 1 (g = 0), beta = 0  =>  S unchanged, o_t = S_0^T q_t."""
    rng = np.random.default_rng(2)
    T, H, d = 7, 2, 5
    q, k, v, g, beta = rand_inputs(rng, T, H, d, d)
    g = np.zeros_like(g)
    beta = np.zeros_like(beta)
    s0 = rng.standard_normal((1, H, d, d))  # not symmetric
    o, s = rec(q, k, v, g, beta, s0)
    want = np.einsum("hij,thi->thj", s0[0], q.astype(np.float64))
    return (np.max(np.abs(s - s0)) <= 1e-14) and (np.max(np.abs(o - want)) <= 1e-12)


def pin_orthonormal_store_recall(rec):
    """alpha = 1, beta = 1, S_0 = 0, keys = d orthonormal vectors: afterwards
    S^T k_j = v_j for every stored pair (an associative memory with no interference)."""
    rng = np.random.default_rng(3)
    d, dv, H = 16, 6, 1
    # rows of a 16x16 Hadamard matrix / 4: orthonormal exactly in binary, then
    # mixed by a random signed permutation
    perm = rng.permutation(d)
    signs = rng.choice([-1.0, 1.0], d)
    keys = f32((hadamard(d) / 4.0)[perm] * signs[:, None])
    T = d
    k = keys.reshape(T, H, d)
    q = k.copy()
    v = f32(rng.standard_normal((T, H, dv)))
    g = np.zeros((T, H, d), np.float32)
    beta = np.ones((T, H), np.float32)
    _, s = rec(q, k, v, g, beta, None)
    K = k[:, 0, :].astype(np.float64)
    V = v[:, 0, :].astype(np.float64)
    err = np.max(np.abs(K @ s[0, 0] - V))
    return err <= 1e-12


def _exact_unrolled(q, k, v, g, beta, s0):
    """Brute force with exact rationals: S_T = (prod A_t) S_0 + sum_t (prod_{s>t} A_s) b_t k_t v_t^T
    with A_t = (I - b_t k_t k_t^T) Diag(a_t) written out as explicit matrices."""
    T, H, dk = q.shape
    dv = v.shape[2]
    outs = np.zeros((T, H, dv))
    finals = np.zeros((H, dk, dv))
    F = Fraction
    for h in range(H):
        A = []
        for t in range(T):
            a = [F(math.exp(float(g[t, h, i]))) for i in range(dk)]
            kk = [F(float(x)) for x in k[t, h]]
            b = F(float(beta[t, h]))
            A.append([[((1 if i == m else 0) - b * kk[i] * kk[m]) * a[m] for m in range(dk)]
                      for i in range(dk)])

        def mm(X, Y):
            return [[sum(X[i][m] * Y[m][j] for m in range(len(Y))) for j in range(len(Y[0]))]
                    for i in range(len(X))]

        S0 = [[F(float(s0[h, i, j])) for j in range(dv)] for i in range(dk)]
        for t in range(T):
            # S_t from the unrolled sum over tokens 0..t
            prod_all = [[F(1 if i == m else 0) for m in range(dk)] for i in range(dk)]
            for s in range(t + 1):
                prod_all = mm(A[s], prod_all)
            St = mm(prod_all, S0)
            for s in range(t + 1):
                P = [[F(1 if i == m else 0) for m in range(dk)] for i in range(dk)]
                for r in range(s + 1, t + 1):
                    P = mm(A[r], P)
                b = F(float(beta[s, h]))
                kv = [[b * F(float(k[s, h, i])) * F(float(v[s, h, j])) for j in range(dv)]
                      for i in range(dk)]
                term = mm(P, kv)
                St = [[St[i][j] + term[i][j] for j in range(dv)] for i in range(dk)]
            qq = [F(float(x)) for x in q[t, h]]
            outs[t, h] = [float(sum(St[i][j] * qq[i] for i in range(dk))) for j in range(dv)]
            if t == T - 1:
                finals[h] = [[float(St[i][j]) for j in range(dv)] for i in range(dk)]
    return outs, finals


def pin_unrolled_brute_force(rec):
    """The sequential recurrence equals the unrolled product-sum, computed exactly."""
    rng = np.random.default_rng(4)
    T, H, d = 5, 2, 3
    q, k, v, g, beta = rand_inputs(rng, T, H, d, d, unit_keys=False)
    s0 = f32(rng.standard_normal((1, H, d, d)))
    o, s = rec(q, k, v, g, beta, s0)
    o_ex, s_ex = _exact_unrolled(q, k, v, g, beta, s0[0])
    return (np.max(np.abs(o - o_ex)) <= 1e-12) and (np.max(np.abs(s[0] - s_ex)) <= 1e-12)


def pin_pure_decay(rec):
    """beta = 0  =>  S_t = Diag(exp(sum_{r<=t} g_r)) S_0 and o_t = S_t^T q_t."""
    rng = np.random.default_rng(5)
    T, H, d = 11, 2, 5
    q, k, v, g, beta = rand_inputs(rng, T, H, d, d, g_lo=-3.0, g_hi=-0.01)
    beta = np.zeros_like(beta)
    s0 = rng.standard_normal((1, H, d, d))
    o, s = rec(q, k, v, g, beta, s0)
    G = np.cumsum(g.astype(np.float64), axis=0)  # [T,H,d]
    St = np.exp(G)[:, :, :, None] * s0[0][None]   # [T,H,dk,dv]
    want_o = np.einsum("thij,thi->thj", St, q.astype(np.float64))
    return (np.max(np.abs(o - want_o)) <= 1e-12) and (np.max(np.abs(s[0] - St[-1])) <= 1e-12)


def pin_lms_step(rec):
    """alpha = 1: one token is one Widrow-Hoff (LMS) step of size beta on
    f(S) = 1/2 |S^T k - v|^2; the gradient here is taken by central finite
    differences, independently of any closed form."""
    rng = np.random.default_rng(6)
    dk, dv, H = 4, 4, 1
    q, k, v, g, beta = rand_inputs(rng, 1, H, dk, dv, unit_keys=False)
    g = np.zeros_like(g)
    s0 = rng.standard_normal((1, H, dk, dv))
    _, s = rec(q, k, v, g, beta, s0)
    kk = k[0, 0].astype(np.float64)
    vv = v[0, 0].astype(np.float64)

    def f(S):
        r = S.T @ kk - vv
        return 0.5 * float(r @ r)

    S = s0[0, 0]
    grad = np.zeros_like(S)
    eps = 1e-6
    for i in range(dk):
        for j in range(dv):
            E = np.zeros_like(S)
            E[i, j] = eps
            grad[i, j] = (f(S + E) - f(S - E)) / (2 * eps)
    want = S - float(beta[0, 0]) * grad
    return np.max(np.abs(s[0, 0] - want)) <= 1e-7


def pin_scalar_geometric(rec):
    """dk = dv = 1 with constant inputs is the first-order recurrence
    S_t = c S_{t-1} + d with c = (1 - b k^2) a, d = b k v, whose closed form is
    S_t = c^t S_0 + d (1 - c^t) / (1 - c); o_t = S_t q."""
    T = 12
    a, b, kk, vv, qq, s0 = 0.5, 0.5, 0.75, 2.0, -1.5, 0.25
    q = np.full((T, 1, 1), qq, np.float32)
    k = np.full((T, 1, 1), kk, np.float32)
    v = np.full((T, 1, 1), vv, np.float32)
    g = np.full((T, 1, 1), math.log(a), np.float32)
    beta = np.full((T, 1), b, np.float32)
    o, s = rec(q, k, v, g, beta, np.full((1, 1, 1, 1), s0))
    a64 = math.exp(float(np.float32(math.log(a))))
    c = (1 - b * kk * kk) * a64
    d = b * kk * vv
    t = np.arange(1, T + 1)
    St = c ** t * s0 + d * (1 - c ** t) / (1 - c)
    return (np.max(np.abs(o[:, 0, 0] - St * qq)) <= 1e-12) and abs(s[0, 0, 0, 0] - St[-1]) <= 1e-12


PINS = [pin_exact_recall, pin_identity, pin_orthonormal_store_recall, pin_unrolled_brute_force,
        pin_pure_decay, pin_lms_step, pin_scalar_geometric]


def _rec(mutation=0):
    def rec(q, k, v, g, beta, s0):
        return oracle.recurrent(q, k, v, g, beta, initial_state=s0, mutation=mutation, nthreads=2)
    return rec


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    assert pin(_rec(0))


@pytest.mark.parametrize("name", sorted(oracle.MUTATIONS))
def test_planted_mistakes_are_caught(name):
    rec = _rec(oracle.MUTATIONS[name])

    def fails(pin):
        try:
            return not pin(rec)
        except RuntimeError:  # mutation not defined for this pin's shapes
            return False

    failed = [p.__name__ for p in PINS if fails(p)]
    assert failed, f"planted mistake '{name}' passed every pin"


def test_non_expansive_with_unit_keys():
    """For |k| = 1, beta in [0,1], alpha in (0,1]: |(I - b k k^T) Diag(a)|_2 <= 1, so
    |S_t|_F <= |S_{t-1}|_F + b |v|; the state stays bounded over long runs."""
    rng = np.random.default_rng(7)
    T, H, d = 200, 2, 8
    q, k, v, g, beta = rand_inputs(rng, T, H, d, d)
    s = rng.standard_normal((1, H, d, d))
    for t in range(T):
        _, s_new = oracle.recurrent(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], beta[t:t + 1],
                                    initial_state=s, nthreads=1)
        for h in range(H):
            lhs = np.linalg.norm(s_new[0, h])
            rhs = np.linalg.norm(s[0, h]) + float(beta[t, h]) * np.linalg.norm(v[t, h].astype(np.float64))
            assert lhs <= rhs + 1e-12
        s = s_new


# ------------------------------------------------------- chunk form (derived)

@pytest.mark.parametrize("C", [16, 32, 64])
@pytest.mark.parametrize("subtile", [False, True])
def test_chunked_equals_recurrent(C, subtile):
    """The chunkwise form with the derived U, W and carry ([K3-notes §2.2,
    chunkwise form]) reproduces the token recurrence, including ragged tails,
    several sequences, random initial states and g = -5 (the decay floor of
    [K3-notes §2.2, Eq. 5])."""
    rng = np.random.default_rng(10 + C)
    lens = [1, 17, C, 2 * C + 5, 0, 3]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, dk, dv = int(cu[-1]), 2, 16, 12
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    g[cu[3]:cu[4]] = -5.0                       # every channel at the floor
    s0 = rng.standard_normal((len(lens), H, dk, dv)) * 0.3
    o_r, s_r = oracle.recurrent(q, k, v, g, beta, s0, cu)
    o_c, s_c = oracle.chunked(q, k, v, g, beta, s0, cu, chunk=C, subtile_ref=subtile)
    assert np.max(np.abs(o_c - o_r)) <= 1e-9 * max(1.0, np.max(np.abs(o_r)))
    assert np.max(np.abs(s_c - s_r)) <= 1e-9 * max(1.0, np.max(np.abs(s_r)))


def test_chunked_diagonal_is_included():
    """A token reads its own write inside a chunk: with beta = 1 and q = k the
    chunk form returns v_t exactly, which needs A's diagonal ([K3-notes §2.2]:
    the causal matrix includes the diagonal)."""
    rng = np.random.default_rng(11)
    T, H, d = 40, 1, 8
    q, k, v, g, beta = rand_inputs(rng, T, H, d, d)
    k = exact_unit_keys(rng, T, H, d)
    q = k.copy()
    beta = np.ones_like(beta)
    o, _ = oracle.chunked(q, k, v, g, beta, rng.standard_normal((1, H, d, d)), chunk=16)
    assert np.max(np.abs(o - v.astype(np.float64))) <= 1e-10


def test_resume_equals_single_run():
    """Prefix-cache resume ([K3-notes §2.5, Fig. 12]): running [0, B) then [B, T)
    from the saved state equals one run over [0, T)."""
    rng = np.random.default_rng(12)
    T, H, dk, dv, Bsplit = 300, 2, 8, 8, 128
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    s0 = rng.standard_normal((1, H, dk, dv))
    o_full, s_full = oracle.recurrent(q, k, v, g, beta, s0)
    o1, s1 = oracle.recurrent(q[:Bsplit], k[:Bsplit], v[:Bsplit], g[:Bsplit], beta[:Bsplit], s0)
    o2, s2 = oracle.chunked(q[Bsplit:], k[Bsplit:], v[Bsplit:], g[Bsplit:], beta[Bsplit:], s1, chunk=64)
    assert np.max(np.abs(np.concatenate([o1, o2]) - o_full)) <= 1e-10
    assert np.max(np.abs(s2 - s_full)) <= 1e-10


def test_varlen_equals_separate_calls():
    rng = np.random.default_rng(13)
    lens = [5, 0, 70, 33]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, dk, dv = int(cu[-1]), 3, 8, 4
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    s0 = rng.standard_normal((len(lens), H, dk, dv))
    o, s = oracle.recurrent(q, k, v, g, beta, s0, cu)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        o_n, s_n = oracle.recurrent(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], s0[n:n + 1])
        assert np.array_equal(s[n], s_n[0])
        assert np.array_equal(o[a:b], o_n)
    # an empty sequence leaves its state as it was
    assert np.array_equal(s[1], s0[1])


def test_chain_subset_matches_full_run():
    rng = np.random.default_rng(14)
    T, H, d = 50, 4, 8
    q, k, v, g, beta = rand_inputs(rng, T, H, d, d)
    o, s = oracle.recurrent(q, k, v, g, beta)
    o2, s2 = oracle.recurrent(q, k, v, g, beta, chains=[1, 3])
    assert np.array_equal(o[:, [1, 3]], o2[:, [1, 3]])
    assert np.all(np.isnan(o2[:, [0, 2]]))
    assert np.array_equal(s[:, [1, 3]], s2[:, [1, 3]])


def test_decode_step_is_one_token():
    rng = np.random.default_rng(15)
    N, H, d = 6, 2, 8
    q, k, v, g, beta = rand_inputs(rng, N, H, d, d)  # one token per sequence
    s0 = rng.standard_normal((N, H, d, d))
    o, s = oracle.decode_step(q, k, v, g, beta, s0)
    cu = np.arange(N + 1)
    o_r, s_r = oracle.recurrent(q, k, v, g, beta, s0, cu)
    assert np.array_equal(o, o_r)
    assert np.array_equal(s, s_r)
    # the closed form of one step (algebra of [K3-notes §2.2] expanded by hand):
    # S' = Diag(a) S + k u^T, u = b (v - S^T (a o k)), o = S^T (a o q) + u (k . q)
    a = np.exp(g.astype(np.float64))
    for n in range(N):
        for h in range(H):
            S = s0[n, h]
            kk, qq, vv = (x[n, h].astype(np.float64) for x in (k, q, v))
            u = float(beta[n, h]) * (vv - S.T @ (a[n, h] * kk))
            assert np.allclose(s[n, h], a[n, h][:, None] * S + np.outer(kk, u), atol=1e-12, rtol=0)
            assert np.allclose(o[n, h], S.T @ (a[n, h] * qq) + u * (kk @ qq), atol=1e-12, rtol=0)


def test_affine_pair_maps_any_entry_state():
    """[K3-notes §2.5]: a segment's effect on its entry state is affine,
    S_out = S~ + M S_in, and pairs compose as (M2 M1, M2 S~1 + S~2)."""
    rng = np.random.default_rng(16)
    T, H, dk, dv = 60, 2, 8, 5
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    h = 1
    M, St = oracle.affine_pair(k, v, g, beta, h, 0, T)
    for _ in range(3):
        s_in = rng.standard_normal((1, H, dk, dv))
        _, s_out = oracle.recurrent(q, k, v, g, beta, s_in)
        assert np.max(np.abs(St + M @ s_in[0, h] - s_out[0, h])) <= 1e-11
    M1, S1 = oracle.affine_pair(k, v, g, beta, h, 0, 23)
    M2, S2 = oracle.affine_pair(k, v, g, beta, h, 23, T)
    assert np.max(np.abs(M2 @ M1 - M)) <= 1e-12
    assert np.max(np.abs(M2 @ S1 + S2 - St)) <= 1e-11
    # one token: M is the explicit transition (I - b k k^T) Diag(a)
    M0, _ = oracle.affine_pair(k, v, g, beta, h, 5, 6)
    kk = k[5, h].astype(np.float64)
    want = (np.eye(dk) - float(beta[5, h]) * np.outer(kk, kk)) @ np.diag(np.exp(g[5, h].astype(np.float64)))
    assert np.max(np.abs(M0 - want)) <= 1e-14


def test_checkpoints_are_prefix_final_states():
    """[K3-notes §2.5, Fig. 12]: the state a request resumes from is the state
    after the shared prefix.  Every recorded checkpoint must equal the final
    state of the recurrence run on that prefix alone (an independent call of
    the pinned token recurrence), and sequences shorter than the interval
    record nothing."""
    rng = np.random.default_rng(11)
    lens = [130, 0, 64, 200, 63]
    every, H, d = 64, 2, 16
    T = sum(lens)
    q = rng.standard_normal((T, H, d)).astype(np.float32)
    k = (q / np.linalg.norm(q, axis=-1, keepdims=True)).astype(np.float32)
    v = rng.standard_normal((T, H, d)).astype(np.float32)
    g = rng.uniform(-0.7, -1e-3, (T, H, d)).astype(np.float32)
    beta = rng.uniform(0, 1, (T, H)).astype(np.float32)
    s0 = rng.standard_normal((len(lens), H, d, d)) * 0.1
    cu = np.concatenate([[0], np.cumsum(lens)])
    _, _, ck, cuc = oracle.recurrent_ckpt(q, k, v, g, beta, every, initial_state=s0, cu_seqlens=cu)
    assert list(np.diff(cuc)) == [n // every for n in lens]
    for n, L in enumerate(lens):
        for j in range(1, L // every + 1):
            rows = slice(cu[n], cu[n] + j * every)
            _, s_pre = oracle.recurrent(q[rows], k[rows], v[rows], g[rows], beta[rows],
                                        initial_state=s0[n:n + 1])
            np.testing.assert_allclose(ck[cuc[n] + j - 1], s_pre[0], rtol=0, atol=1e-12)


def test_resume_from_checkpoint_matches_full_run():
    """Resuming the recurrence from a checkpoint on the rest of the sequence
    gives the full run's outputs and final state (prefix-cache reuse)."""
    rng = np.random.default_rng(12)
    T, H, d, every = 320, 2, 16, 64
    q = rng.standard_normal((T, H, d)).astype(np.float32)
    k = (q / np.linalg.norm(q, axis=-1, keepdims=True)).astype(np.float32)
    v = rng.standard_normal((T, H, d)).astype(np.float32)
    g = rng.uniform(-0.7, -1e-3, (T, H, d)).astype(np.float32)
    beta = rng.uniform(0, 1, (T, H)).astype(np.float32)
    o, sf, ck, _ = oracle.recurrent_ckpt(q, k, v, g, beta, every)
    for j in (1, 3):
        cut = j * every
        o2, s2 = oracle.recurrent(q[cut:], k[cut:], v[cut:], g[cut:], beta[cut:], initial_state=ck[j - 1:j])
        np.testing.assert_allclose(o2, o[cut:], rtol=0, atol=1e-10)
        np.testing.assert_allclose(s2, sf, rtol=0, atol=1e-10)


def test_state_columns_split_equals_full_run():
    """Column j of the state is written by entry j of v alone ([K3-notes §2.2]:
    the erase and the decay act on S from the left), so running a head as
    independent chains of a few state columns gives the full run exactly.
    The long-context parity test relies on this to spread one 2^20-token head
    over several host cores."""
    from _helpers import oracle_heads_by_columns
    from hybrid_linear_attention_chunk_gb300 import inputs
    w = inputs.scaled(inputs.LONG_T1M, B=1, T=0, H=3, dk=16, dv=16, varlen_seqs=3, len_lo=20, len_hi=90)
    x = inputs.make_prefill(w, lengths=np.array([70, 0, 45]))
    h = {n: inputs.host_f32(x[n]) for n in ("q", "k", "v", "log_alpha", "beta", "initial_state")}
    cu = x["cu_seqlens"].numpy()
    o, s = oracle.recurrent(h["q"], h["k"], h["v"], h["log_alpha"], h["beta"], h["initial_state"], cu)
    o2, s2 = oracle_heads_by_columns(x, [2, 0], width=4, workers=3)
    assert np.array_equal(o2, o[:, [2, 0]]) and np.array_equal(s2, s[:, [2, 0]])
