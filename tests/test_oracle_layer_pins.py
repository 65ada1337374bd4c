"""Pins for the oracle's KDA layer gates (``oracle.layer``, ``oracle.layer_decode_step``).

Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
(liuzhao09.github.io/papers/kimi-k3), [K3-notes] below.
  [K3-notes §2.2, Eq. 5]:            g = g_min Sigmoid(exp(A_h) z),  alpha = exp(g)
  [K3-notes §2.2, KDA output]:       y = Sigmoid(W_g x) o RMSNorm(o~)   (per head)
RMSNorm(x)_j = x_j w_j / sqrt(mean x^2 + eps) (the page names the norm only).

The pins read the gates through the recurrence with inputs that make it
transparent: one token with q = k = e_0 and beta = 1 from a zero state gives
o~ = v exactly, and a second token that writes nothing (beta = 0) and reads
along e_0 gives o~ = alpha_0 v, so the decay of channel 0 is visible.  The
expected values are closed forms; ``test_planted_gate_mistakes_are_caught``
plants each plausible slip in the oracle and checks that a pin fails.
"""
import math

import numpy as np
import pytest

import oracle


def f32(x):
    return np.asarray(x, dtype=np.float32)


def decay_probe(z0, A, g_min, H=1, mutation=0):
    """alpha of channel 0 at token 2 for each head, read through the recurrence.

    z0: [H] logits of channel 0 at token 2; A: [H]."""
    dk = dv = 4
    q = np.zeros((2, H, dk)); k = np.zeros((2, H, dk)); v = np.zeros((2, H, dv))
    q[:, :, 0] = 1.0
    k[0, :, 0] = 1.0
    k[1, :, 1] = 1.0
    v[0, :, :] = [1.0, 2.0, -3.0, 0.5]
    beta = np.zeros((2, H)); beta[0] = 1.0
    z = np.zeros((2, H, dk)); z[1, :, 0] = z0
    o, _ = oracle.layer(f32(q), f32(k), f32(v), f32(z), f32(beta), f32(A), g_min=g_min, mutation=mutation)
    return o[1, :, 0], o[1, :, 1] / 2.0


def norm_probe(v_row, gate_row, w=None, eps=0.0, mutation=0):
    """One token whose o~ is v_row exactly, through the output norm and gate."""
    dv = len(v_row)
    q = np.zeros((1, 1, 4)); k = np.zeros((1, 1, 4))
    q[0, 0, 0] = k[0, 0, 0] = 1.0
    v = np.asarray(v_row, np.float64).reshape(1, 1, dv)
    z = np.zeros((1, 1, 4))
    o, _ = oracle.layer(f32(q), f32(k), f32(v), f32(z), f32(np.ones((1, 1))), f32([0.0]),
                        out_gate=f32(np.asarray(gate_row).reshape(1, 1, dv)),
                        norm_weight=None if w is None else f32(w), norm_eps=eps, mutation=mutation)
    return o[0, 0]


# ------------------------------------------------------------------ pins

def pin_decay_zero_logit(mut):
    """z = 0: Sigmoid(0) = 1/2, so alpha = exp(g_min / 2) whatever A is."""
    a0, a1 = decay_probe([0.0], [0.7], -5.0, mutation=mut)
    return np.allclose(a0, math.exp(-2.5), rtol=1e-12) and np.allclose(a1, math.exp(-2.5), rtol=1e-12)


def pin_decay_three_quarters(mut):
    """exp(A) z = ln 3 gives Sigmoid = 3/4: head 0 with A = 0, z = ln 3; head 1
    with A = ln 2, z = ln 3 / 2 (the fp32 rounding of the inputs moves alpha
    by < 1e-6 relative)."""
    a0, _ = decay_probe([math.log(3.0), math.log(3.0) / 2], [0.0, math.log(2.0)], -4.0, H=2, mutation=mut)
    return np.allclose(a0, math.exp(-3.0), rtol=1e-6)


def pin_decay_saturates(mut):
    """z -> +inf: alpha -> exp(g_min) (the floor of Eq. 5); z -> -inf: alpha -> 1."""
    hi, _ = decay_probe([60.0], [0.0], -2.0, mutation=mut)
    lo, _ = decay_probe([-60.0], [0.0], -2.0, mutation=mut)
    return np.allclose(hi, math.exp(-2.0), rtol=1e-12) and np.allclose(lo, 1.0, rtol=1e-12)


def pin_norm_worked_example(mut):
    """o~ = (3, 4): mean square 12.5, so RMSNorm = (3, 4) / (5 / sqrt 2); gates
    0 and ln 3 give Sigmoid 1/2 and 3/4: y = (3 sqrt2 / 10, 3 sqrt2 / 5)."""
    y = norm_probe([3.0, 4.0], [0.0, math.log(3.0)], mutation=mut)
    r2 = math.sqrt(2.0)
    return np.allclose(y, [3 * r2 / 10, 3 * r2 / 5], rtol=1e-6)


def pin_norm_weight(mut):
    """A per-channel weight (2, -1) scales channel by channel."""
    r2 = math.sqrt(2.0)
    y = norm_probe([3.0, 4.0], [60.0, 60.0], w=[2.0, -1.0], mutation=mut)
    return np.allclose(y, [2 * 3 * r2 / 5, -4 * r2 / 5], rtol=1e-12)


def pin_norm_eps(mut):
    """eps = 37.5 adds to the mean square 12.5: the divisor is sqrt 50 = 5 sqrt 2."""
    y = norm_probe([3.0, 4.0], [60.0, 60.0], eps=37.5, mutation=mut)
    return np.allclose(y, [3 / (5 * math.sqrt(2.0)), 4 / (5 * math.sqrt(2.0))], rtol=1e-12)


def pin_norm_unit_rms_scale_free(mut):
    """With the gate open (Sigmoid = 1), w = 1 and eps = 0 the output has RMS 1
    and does not change when o~ is scaled."""
    rng = np.random.default_rng(3)
    v = rng.standard_normal(128)
    y1 = norm_probe(v, np.full(128, 60.0), mutation=mut)
    y2 = norm_probe(8.0 * v, np.full(128, 60.0), mutation=mut)
    return abs(np.sqrt(np.mean(y1 ** 2)) - 1.0) < 1e-12 and np.allclose(y1, y2, rtol=1e-12, atol=0)


PINS = [pin_decay_zero_logit, pin_decay_three_quarters, pin_decay_saturates, pin_norm_worked_example,
        pin_norm_weight, pin_norm_eps, pin_norm_unit_rms_scale_free]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_gate_pin(pin):
    assert pin(0)


@pytest.mark.parametrize("name", sorted(oracle.GATE_MUTATIONS))
def test_planted_gate_mistakes_are_caught(name):
    mut = oracle.GATE_MUTATIONS[name]
    assert not all(p(mut) for p in PINS), f"no pin catches the planted slip {name}"


# ------------------------------------------------------- layer = recurrence

def test_layer_is_the_recurrence_with_the_gate_decay():
    """With the output gate off, the layer is the plain recurrence run on the
    log-decay that Eq. 5 gives; every head uses its own A_h."""
    rng = np.random.default_rng(11)
    T, H, dk, dv = 37, 3, 8, 6
    q = rng.standard_normal((T, H, dk)); k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    z = 3.0 * rng.standard_normal((T, H, dk))
    A = rng.uniform(-1.0, 1.0, H)
    beta = rng.uniform(0.0, 1.0, (T, H))
    s0 = rng.standard_normal((2, H, dk, dv))
    cu = np.array([0, 20, 37])
    q, k, v, z, A, beta = (f32(x) for x in (q, k, v, z, A, beta))
    g = -5.0 / (1.0 + np.exp(-np.exp(A.astype(np.float64))[None, :, None] * z.astype(np.float64)))
    o_l, s_l = oracle.layer(q, k, v, z, beta, A, -5.0, initial_state=s0, cu_seqlens=cu)
    # the plain recurrence takes fp32 log-decay: compare at that rounding
    o_r, s_r = oracle.recurrent(q, k, v, f32(g), beta, s0, cu)
    assert np.allclose(o_l, o_r, rtol=1e-5, atol=1e-6)
    assert np.allclose(s_l, s_r, rtol=1e-5, atol=1e-6)
    assert np.all(g > -5.0) and np.all(g < 0.0)  # Eq. 5 keeps the log-decay in (g_min, 0)


def test_layer_output_gate_acts_row_by_row():
    """The output gate and norm change only the outputs, token by token: the
    states match the ungated run, and each output row is the ungated row
    normalised over its dv channels and gated."""
    rng = np.random.default_rng(12)
    T, H, dk, dv = 21, 2, 8, 16
    q = f32(rng.standard_normal((T, H, dk))); k = rng.standard_normal((T, H, dk))
    k = f32(k / np.linalg.norm(k, axis=-1, keepdims=True))
    v = f32(rng.standard_normal((T, H, dv))); z = f32(rng.standard_normal((T, H, dk)))
    A = f32([0.3, -0.4]); beta = f32(rng.uniform(0, 1, (T, H)))
    gate = f32(2.0 * rng.standard_normal((T, H, dv))); w = f32(rng.uniform(0.5, 1.5, dv))
    o0, s0 = oracle.layer(q, k, v, z, beta, A)
    o1, s1 = oracle.layer(q, k, v, z, beta, A, out_gate=gate, norm_weight=w, norm_eps=1e-5)
    assert np.array_equal(s0, s1)
    # ratio o1 / o0 per row: Sigmoid(gate) w / rms, with one rms per (token, head)
    ratio = o1 / o0 / (w[None, None, :] / (1.0 + np.exp(-gate.astype(np.float64))))
    assert np.allclose(ratio, ratio[:, :, :1], rtol=1e-10)
    rms = np.sqrt(np.mean(o0 ** 2, axis=-1, keepdims=True) + 1e-5)
    assert np.allclose(ratio[:, :, :1], 1.0 / rms, rtol=1e-10)


def test_layer_decode_step_is_one_layer_token():
    rng = np.random.default_rng(13)
    N, H, dk, dv = 3, 2, 8, 8
    q, k, v, z, gate = (f32(rng.standard_normal((N, H, d))) for d in (dk, dk, dv, dk, dv))
    k = f32(k / np.linalg.norm(k, axis=-1, keepdims=True))
    beta = f32(rng.uniform(0, 1, (N, H))); A = f32([0.1, -0.2])
    S = rng.standard_normal((N, H, dk, dv))
    o_d, S_d = oracle.layer_decode_step(q, k, v, z, beta, S, A, -5.0, out_gate=gate, norm_eps=1e-6)
    o_l, S_l = oracle.layer(q, k, v, z, beta, A, -5.0, out_gate=gate, norm_eps=1e-6, initial_state=S,
                            cu_seqlens=np.arange(N + 1))
    assert np.array_equal(o_d, o_l) and np.array_equal(S_d, S_l)
