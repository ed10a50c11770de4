"""Pins for the oracle's state functions (the stateful / cross-attention
extension of the forward pass): each is checked against an independently
pinned oracle form, a brute-force loop on tiny inputs, or an invariant."""
import math

import numpy as np
import pytest

import oracle as O
from synth import make_omega_orf


def _inputs(seed, B=2, H=2, Lq=37, Lk=37, d=8, dv=5, m=16):
    rng = np.random.default_rng(seed)
    q = rng.normal(size=(B, H, Lq, d)) * 0.5
    k = rng.normal(size=(B, H, Lk, d)) * 0.5
    v = rng.normal(size=(B, H, Lk, dv))
    omega = np.stack([make_omega_orf(rng, m, d) for _ in range(H)])
    return q, k, v, omega


@pytest.mark.parametrize("kind", O.KINDS)
def test_state_then_readout_equals_bidirectional(kind):
    q, k, v, om = _inputs(1)
    s = 0.7
    got = O.favor_attn_from_state(q, O.favor_kv_state(k, v, om, s, kind), om, s, kind)
    ref = O.favor_bidir(q, k, v, om, s, kind)
    assert np.max(np.abs(got - ref)) < 1e-12


@pytest.mark.parametrize("kind", O.KINDS)
def test_cross_attention_brute_force(kind):
    # Lq != Lk: a loop over queries, keys and features with scalar math
    q, k, v, om = _inputs(2, B=1, H=1, Lq=4, Lk=6, d=3, dv=2, m=5)
    s = 0.9
    got = O.favor_attn_from_state(q, O.favor_kv_state(k, v, om, s, kind), om, s, kind)[0, 0]
    w = om[0]

    def phi(x):
        out = []
        for r in range(w.shape[0]):
            p = sum(w[r, c] * s * x[c] for c in range(len(x)))
            if kind == "softmax_pos":
                out.append(math.exp(p - 0.5 * sum((s * t) ** 2 for t in x)) / math.sqrt(w.shape[0]))
            else:
                out.append(max(p, 0.0) / math.sqrt(w.shape[0]))
        return out

    for i in range(4):
        fq = phi(q[0, 0, i])
        num = [0.0, 0.0]
        den = 0.0
        for j in range(6):
            fk = phi(k[0, 0, j])
            a = sum(x * y for x, y in zip(fq, fk))
            den += a
            num = [num[e] + a * v[0, 0, j, e] for e in range(2)]
        ref = [x / den for x in num] if den != 0.0 else [0.0, 0.0]
        assert np.allclose(got[i], ref, rtol=1e-12, atol=1e-14)


def test_state_is_linear_in_the_keys():
    q, k, v, om = _inputs(3, Lk=30)
    s = 0.8
    a = O.favor_kv_state(k[:, :, :11], v[:, :, :11], om, s)
    b = O.favor_kv_state(k[:, :, 11:], v[:, :, 11:], om, s)
    assert np.max(np.abs(a + b - O.favor_kv_state(k, v, om, s))) < 1e-12


@pytest.mark.parametrize("kind", O.KINDS)
def test_causal_from_state_chained_equals_causal(kind):
    q, k, v, om = _inputs(4, Lq=50, Lk=50)
    s = 0.75
    state = np.zeros(k.shape[:2] + (om.shape[1], v.shape[-1] + 1))
    outs = []
    t0 = 0
    for T in (1, 7, 20, 22):
        o, state = O.favor_causal_from_state(q[:, :, t0:t0 + T], k[:, :, t0:t0 + T], v[:, :, t0:t0 + T],
                                             state, om, s, kind)
        outs.append(o)
        t0 += T
    got = np.concatenate(outs, axis=2)
    assert np.max(np.abs(got - O.favor_causal(q, k, v, om, s, kind))) < 1e-12
    assert np.max(np.abs(state - O.favor_kv_state(k, v, om, s, kind))) < 1e-12
    # and the token-by-token recurrence, one head
    pq = O.feature_map(s * q[1, 0], om[0], kind)
    pk = O.feature_map(s * k[1, 0], om[0], kind)
    assert np.max(np.abs(got[1, 0] - O.rnn_causal_from_features(pq, pk, v[1, 0]))) < 1e-12
