"""Pins for the oracle's feature-map variants: hyperbolic positive features
(SM^hyp+), trigonometric features (SM^trig) and regularized projections
(SMREG), from Rethinking Attention with Performers §2.3, Lemma 1 and Lemma 2.

Each pin compares the oracle with a closed form written through another route
(hyperbolic cosine, angle-difference identity, Bessel-function spherical
means), a Monte Carlo law, or a structural fact of the projections.
"""
import math

import numpy as np
import pytest

import oracle as O
from synth import make_omega_iid, make_omega_orf


def _xy():
    x = np.array([0.3, -0.2, 0.1, 0.4, 0.0, -0.1])
    y = np.array([-0.1, 0.25, 0.3, 0.2, -0.3, 0.05])
    return x, y


def test_hyperbolic_inner_product_is_cosh_estimate():
    """phi_hyp(x).phi_hyp(y) = Lambda (1/M) sum_r cosh(omega_r . (x + y)) with
    Lambda = exp(-(||x||^2 + ||y||^2)/2): the hyperbolic-cosine form of Eq. 7."""
    rng = np.random.default_rng(1)
    x, y = _xy()
    om = rng.standard_normal((7, 6))
    lam = math.exp(-0.5 * (x @ x + y @ y))
    ref = lam * sum(math.cosh(float(w @ (x + y))) for w in om) / len(om)
    got = float(O.feature_map_hyperbolic(x[None], om)[0] @ O.feature_map_hyperbolic(y[None], om)[0])
    assert got == pytest.approx(ref, rel=1e-13)
    assert O.feature_map_hyperbolic(x[None], om).shape == (1, 14)
    assert np.all(O.feature_map_hyperbolic(x[None], om) > 0)


def test_trig_inner_product_is_gaussian_kernel_estimate():
    """phi_trig(x).phi_trig(y) = exp((||x||^2 + ||y||^2)/2) (1/M) sum_r cos(omega_r . (x - y)):
    sin a sin b + cos a cos b = cos(a - b), the random Fourier estimate of the
    Gaussian kernel scaled by h(x) h(y) (§2.3)."""
    rng = np.random.default_rng(2)
    x, y = _xy()
    om = rng.standard_normal((9, 6))
    ref = math.exp(0.5 * (x @ x + y @ y)) * sum(math.cos(float(w @ (x - y))) for w in om) / len(om)
    got = float(O.feature_map_trig(x[None], om)[0] @ O.feature_map_trig(y[None], om)[0])
    assert got == pytest.approx(ref, rel=1e-13)


@pytest.mark.parametrize("kind", O.VARIANT_KINDS)
def test_variant_estimators_unbiased_with_lemma2_mse(kind):
    """Monte Carlo over single-draw estimators (M = 1, iid Gaussian omega):
    mean -> exp(x.y) and the MSE matches Lemma 2:
        trig: (1/2M) exp(||x||^2 + ||y||^2) (1 - exp(-||x - y||^2))^2
        hyp+: (1/2)(1 - exp(-||x + y||^2)) * MSE(SM+),
              MSE(SM+) = (1/M) exp(||x+y||^2) SM(x,y)^2 (1 - exp(-||x+y||^2))."""
    rng = np.random.default_rng(3)
    x, y = _xy()
    sm = math.exp(x @ y)
    zz = float((x + y) @ (x + y))
    dd = float((x - y) @ (x - y))
    if kind == "softmax_trig":
        mse = 0.5 * math.exp(x @ x + y @ y) * (1 - math.exp(-dd)) ** 2
    else:
        mse = 0.5 * (1 - math.exp(-zz)) * math.exp(zz) * sm ** 2 * (1 - math.exp(-zz))
    n = 400_000
    om = rng.standard_normal((n, 6))
    px = O.feature_map(x[None], om, kind)[0]
    py = O.feature_map(y[None], om, kind)[0]
    # one M = 1 estimate per row r: features r and r + n, rescaled from M = n to M = 1
    est = n * (px[:n] * py[:n] + px[n:] * py[n:])
    assert abs(est.mean() - sm) < 5 * math.sqrt(mse / n)
    assert np.mean((est - sm) ** 2) == pytest.approx(mse, rel=0.05)


def test_hyperbolic_beats_positive_with_same_draws():
    """Lemma 2: MSE(hyp+) = (1/2)(1 - exp(-||x+y||^2)) MSE(SM+) < MSE(SM+)/2 for the
    same number M of draws; checked empirically with M = 4 over many draws."""
    rng = np.random.default_rng(4)
    x, y = _xy()
    sm = math.exp(x @ y)
    errs_pos, errs_hyp = [], []
    for _ in range(20000):
        om = rng.standard_normal((4, 6))
        ep = float(O.feature_map_positive(x[None], om)[0] @ O.feature_map_positive(y[None], om)[0])
        eh = float(O.feature_map_hyperbolic(x[None], om)[0] @ O.feature_map_hyperbolic(y[None], om)[0])
        errs_pos.append((ep - sm) ** 2)
        errs_hyp.append((eh - sm) ** 2)
    zz = float((x + y) @ (x + y))
    ratio = np.mean(errs_hyp) / np.mean(errs_pos)
    assert ratio == pytest.approx(0.5 * (1 - math.exp(-zz)), rel=0.1)


def test_hyperbolic_equals_positive_with_mirrored_rows():
    """exp(-omega.x) = exp((-omega).x): the hyperbolic map of omega is the positive
    map of the 2M rows [omega; -omega] (same 1/sqrt(2M) factor)."""
    rng = np.random.default_rng(5)
    x = rng.normal(0, 0.5, (11, 8))
    om = rng.standard_normal((6, 8))
    np.testing.assert_allclose(O.feature_map_hyperbolic(x, om),
                               O.feature_map_positive(x, np.concatenate([om, -om])), rtol=1e-14)


def test_trig_attention_brute_force():
    """Bidirectional and causal attention with trigonometric features against
    explicit loops over (i, j) of phi_trig(q_i).phi_trig(k_j) built from the
    angle-difference form (any sign: no zero-denominator row here)."""
    rng = np.random.default_rng(6)
    L, d, dv, M = 7, 4, 3, 5
    om = rng.standard_normal((1, M, d))
    q, k = rng.normal(0, 0.4, (1, 1, L, d)), rng.normal(0, 0.4, (1, 1, L, d))
    v = rng.normal(0, 1, (1, 1, L, dv))
    for causal in (False, True):
        a = np.zeros((L, L))
        for i in range(L):
            for j in range(L):
                if causal and j > i:
                    continue
                xi, yj = q[0, 0, i], k[0, 0, j]
                a[i, j] = math.exp(0.5 * (xi @ xi + yj @ yj)) * sum(
                    math.cos(float(w @ (xi - yj))) for w in om[0]) / M
        ref = (a @ v[0, 0]) / a.sum(1, keepdims=True)
        fn = O.favor_causal if causal else O.favor_bidir
        np.testing.assert_allclose(fn(q, k, v, om, 1.0, "softmax_trig")[0, 0], ref, rtol=1e-11)


def test_smreg_rows_have_length_sqrt_d_and_stay_orthogonal():
    rng = np.random.default_rng(7)
    d = 16
    om = make_omega_orf(rng, 48, d, regularized=True)
    np.testing.assert_allclose(np.linalg.norm(om, axis=1), math.sqrt(d), rtol=1e-13)
    for b in range(3):
        blk = om[b * d:(b + 1) * d]
        np.testing.assert_allclose(blk @ blk.T, d * np.eye(d), atol=1e-12)
    iid = make_omega_iid(rng, 40, d, regularized=True)
    np.testing.assert_allclose(np.linalg.norm(iid, axis=1), math.sqrt(d), rtol=1e-13)


def test_smreg_estimate_matches_spherical_mean_and_lower_bounds_softmax():
    """With D = Unif(sqrt(d) S^{d-1}) the positive estimator is unbiased for
    SMREG(x, y) = Lambda E_u[exp(sqrt(d) u.(x+y))] = Lambda Gamma(d/2) (t/2)^{1-d/2} I_{d/2-1}(t),
    t = sqrt(d) ||x+y|| (the spherical mean of an exponential), and
    SMREG <= SM (Theorem 1: the regularized kernel is a lower bound)."""
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(8)
    x, y = _xy()
    d = 6
    z = x + y
    t = math.sqrt(d) * math.sqrt(float(z @ z))
    nu = d / 2 - 1
    sph = math.exp(math.lgamma(d / 2) + (1 - d / 2) * math.log(t / 2) + t) * float(special.ive(nu, t))
    smreg = math.exp(-0.5 * (x @ x + y @ y)) * sph
    assert smreg <= math.exp(x @ y)
    n = 400_000
    om = make_omega_iid(rng, n, d, regularized=True)
    est = n * O.feature_map_positive(x[None], om)[0] * O.feature_map_positive(y[None], om)[0]
    assert abs(est.mean() - smreg) < 5 * est.std() / math.sqrt(n)
