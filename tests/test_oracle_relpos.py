"""Pins for the oracle's gated causal attention (RFA-Gate) and PermuteFormer
relative-position attention: special cases with known outputs and explicit
L x L forms built by loops through a different route than the oracle's."""
import numpy as np
import pytest

import oracle as O
from synth import make_omega_orf


def _case(seed, L=13, d=4, dv=3, m=8, H=2, B=1):
    rng = np.random.default_rng(seed)
    omega = np.stack([make_omega_orf(rng, m, d) for _ in range(H)])
    q = rng.normal(0, 0.5, (B, H, L, d))
    k = rng.normal(0, 0.5, (B, H, L, d))
    v = rng.normal(0, 1.0, (B, H, L, dv))
    return rng, omega, q, k, v


# ------------------------------------------------------------------ RFA-Gate
def test_gate_zero_attends_to_the_current_token_only():
    """g = 0 keeps only phi(k_t) v_t^T: out_t = v_t for positive features."""
    _, omega, q, k, v = _case(1)
    g = np.zeros(q.shape[:3])
    np.testing.assert_allclose(O.favor_causal_gated(q, k, v, g, omega, 0.9), v, rtol=1e-12)


def test_gate_one_never_writes_the_state():
    """g = 1 keeps S = 0 and z = 0: every denominator is 0, every row is 0."""
    _, omega, q, k, v = _case(2)
    g = np.ones(q.shape[:3])
    np.testing.assert_array_equal(O.favor_causal_gated(q, k, v, g, omega, 0.9), 0.0)


def test_gate_matches_explicit_weights():
    """Unrolling the recurrence: out_t = sum_j w_tj A_tj v_j / sum_j w_tj A_tj with
    w_tj = (1 - g_j) prod_{l=j+1..t} g_l and A_tj = phi(q_t).phi(k_j), j <= t;
    built by explicit loops."""
    rng, omega, q, k, v = _case(3, L=11)
    g = rng.uniform(0.2, 0.95, q.shape[:3])
    got = O.favor_causal_gated(q, k, v, g, omega, 0.8)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            pq = O.feature_map(0.8 * q[b, h], omega[h], "softmax_pos")
            pk = O.feature_map(0.8 * k[b, h], omega[h], "softmax_pos")
            L = pq.shape[0]
            for t in range(L):
                num = np.zeros(v.shape[-1])
                den = 0.0
                for j in range(t + 1):
                    w = 1.0 - g[b, h, j]
                    for l in range(j + 1, t + 1):
                        w *= g[b, h, l]
                    a = float(pq[t] @ pk[j])
                    num += w * a * v[b, h, j]
                    den += w * a
                np.testing.assert_allclose(got[b, h, t], num / den, rtol=1e-11)


def test_constant_gate_is_exponentially_decayed_attention():
    """A constant gate g: the common (1 - g) cancels and the weights are g^(t-j)
    (tril of a Toeplitz decay matrix times the kernel estimates)."""
    _, omega, q, k, v = _case(4, L=20)
    g = 0.7
    got = O.favor_causal_gated(q, k, v, np.full(q.shape[:3], g), omega, 0.8)
    pq = O.feature_map(0.8 * q[0, 0], omega[0], "softmax_pos")
    pk = O.feature_map(0.8 * k[0, 0], omega[0], "softmax_pos")
    idx = np.arange(20)
    decay = np.tril(g ** (idx[:, None] - idx[None, :]).clip(min=0))
    a = (pq @ pk.T) * decay
    np.testing.assert_allclose(got[0, 0], (a @ v[0, 0]) / a.sum(1, keepdims=True), rtol=1e-11)


# ------------------------------------------------------------------ PermuteFormer
def _inverse(perm):
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    return inv


def _power_by_cycles(perm, n):
    """pi^n for any integer n via the cycle decomposition (a different route
    than repeated indexing): each element moves n steps along its cycle."""
    m = len(perm)
    out = np.empty(m, dtype=int)
    seen = np.zeros(m, dtype=bool)
    for a0 in range(m):
        if seen[a0]:
            continue
        cyc = [a0]
        seen[a0] = True
        b = perm[a0]
        while b != a0:
            cyc.append(b)
            seen[b] = True
            b = perm[b]
        for t, a in enumerate(cyc):
            out[a] = cyc[(t + n) % len(cyc)]
    return out


def test_identity_permutation_and_unit_decay_is_performer():
    _, omega, q, k, v = _case(5)
    perm = np.tile(np.arange(8), (2, 1))
    for causal in (False, True):
        got = O.favor_permute(q, k, v, omega, 0.8, perm, np.ones(2), causal)
        ref = (O.favor_causal if causal else O.favor_bidir)(q, k, v, omega, 0.8)
        np.testing.assert_allclose(got, ref, rtol=1e-12)


def test_permutation_power_by_indexing_matches_cycles():
    rng = np.random.default_rng(6)
    perm = rng.permutation(12)
    for n in range(0, 30, 7):
        np.testing.assert_array_equal(O.permutation_power(perm, n), _power_by_cycles(perm, n))


@pytest.mark.parametrize("causal", [False, True])
def test_permuteformer_matches_relative_position_similarity(causal):
    """sim(i, j) = r^(i-j) sum_b phi(q_i)_b phi(k_j)_{pi^(j-i)(b)}: the similarity
    depends on i - j only ([PF] Property 1); built by loops with powers from the
    cycle decomposition (negative powers for j < i)."""
    rng, omega, q, k, v = _case(7, L=10, m=8)
    perm = np.stack([rng.permutation(8) for _ in range(2)])
    r = np.array([0.9, 0.75])
    got = O.favor_permute(q, k, v, omega, 0.8, perm, r, causal)
    for h in range(2):
        pq = O.feature_map(0.8 * q[0, h], omega[h], "softmax_pos")
        pk = O.feature_map(0.8 * k[0, h], omega[h], "softmax_pos")
        L = pq.shape[0]
        rr = r[h] if causal else 1.0
        for i in range(L):
            num = np.zeros(v.shape[-1])
            den = 0.0
            for j in range(L):
                if causal and j > i:
                    continue
                pw = _power_by_cycles(perm[h], j - i)
                sim = rr ** (i - j) * sum(pq[i, b] * pk[j, pw[b]] for b in range(8))
                num += sim * v[0, h, j]
                den += sim
            np.testing.assert_allclose(got[0, h, i], num / den, rtol=1e-10)


def test_permutation_order_period():
    """A single m-cycle has order m: P^m = I, so query i and key i + m (bidir,
    r = 1) pair feature b with feature b, exactly as at distance 0."""
    m = 8
    perm = np.roll(np.arange(m), 1)             # one cycle of length 8
    assert np.array_equal(O.permutation_power(perm, m), np.arange(m))
    phi = np.random.default_rng(8).random((2 * m + 1, m))
    a = O.permute_features(phi, perm, 1.0, +1)
    np.testing.assert_allclose(a[m], phi[m])
    np.testing.assert_allclose(a[2 * m], phi[2 * m])
    np.testing.assert_allclose(a[1], phi[1][perm])
