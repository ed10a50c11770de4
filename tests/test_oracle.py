"""Pins for the float64 oracle, checked against what the pages and mathematics fix.

None of these tests retypes an oracle formula: each compares the oracle with a
printed value, a hand-computed literal, a brute-force loop on tiny inputs, a
closed form, an invariant, or a statistical law from the pages.
"""
import math
import os

import numpy as np
import pytest

import oracle as O
from synth import make_omega_iid, make_omega_orf, round_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, val = (t.strip() for t in line.split("=", 1))
        vals[key] = np.array([[float(x) for x in row.split()] for row in val.split(";")])
    return vals


# ---------------------------------------------------------------- worked example
def test_worked_example_bidirectional():
    """Performer explainer §2 teaching example: S=(3,10), z=(1,2), output 13/3."""
    g = _read_golden("worked_example.txt")
    pk, v, pq = g["key_features"], g["values"], g["query_feature"]
    s, z = O.bidir_state(pk, v)
    np.testing.assert_array_equal(s, g["S"])
    np.testing.assert_array_equal(z, g["z"].ravel())
    out = O.attn_from_features_bidir(pq, pk, v)
    assert out.shape == (1, 1)
    assert out[0, 0] == pytest.approx(g["output_num"][0, 0] / g["output_den"][0, 0], rel=1e-15)
    # the same output as a weighted average with the printed weights 1 and 2
    w = g["weights"].ravel()
    assert out[0, 0] == pytest.approx((w @ v.ravel()) / w.sum(), rel=1e-15)


def test_worked_example_causal():
    """Causal form of the same example: query (1,1) at both positions.
    Row 1 sees only key 1 (weight 1, value 3); row 2 sees both (13/3)."""
    g = _read_golden("worked_example.txt")
    pk, v = g["key_features"], g["values"]
    pq = np.repeat(g["query_feature"], 2, axis=0)
    out = O.attn_from_features_causal(pq, pk, v)
    assert out[0, 0] == pytest.approx(3.0, rel=1e-15)
    assert out[1, 0] == pytest.approx(13.0 / 3.0, rel=1e-15)


# ------------------------------------------------------ reordering vs brute force
def _brute(pq, pk, v, causal):
    """L x L attention by explicit loops (Eq. 1/2 with the kernel estimate)."""
    L, dv = pq.shape[0], v.shape[1]
    out = np.zeros((L, dv))
    for i in range(L):
        num = np.zeros(dv)
        den = 0.0
        for j in range(pk.shape[0]):
            if causal and j > i:
                continue
            a = sum(pq[i, r] * pk[j, r] for r in range(pq.shape[1]))
            num += a * v[j]
            den += a
        out[i] = num / den
    return out


def test_associativity_4x3x2():
    """Explainer §2: 4 tokens, feature width 3, value width 2 -- the reordered
    product equals the explicit 4 x 4 path."""
    rng = np.random.default_rng(11)
    pq, pk = rng.uniform(0.1, 2.0, (4, 3)), rng.uniform(0.1, 2.0, (4, 3))
    v = rng.standard_normal((4, 2))
    np.testing.assert_allclose(O.attn_from_features_bidir(pq, pk, v), _brute(pq, pk, v, False),
                               rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(O.attn_from_features_causal(pq, pk, v), _brute(pq, pk, v, True),
                               rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_favor_vs_brute_force_tiny(causal):
    """Whole path (features + attention) against loops at L=9, d=4, m=8."""
    rng = np.random.default_rng(5)
    L, d, m = 9, 4, 8
    q, k, v = rng.normal(0, .5, (L, d)), rng.normal(0, .5, (L, d)), rng.normal(0, 1, (L, 3))
    om = rng.standard_normal((m, d))
    s = 0.7
    # features by loops with math.exp, from Lemma 1's per-feature formula
    def phi(x):
        x = s * x
        return np.array([[math.exp(sum(om[r, c] * x[i, c] for c in range(d))
                                   - 0.5 * sum(x[i, c] ** 2 for c in range(d))) / math.sqrt(m)
                          for r in range(m)] for i in range(L)])
    ref = _brute(phi(q), phi(k), v, causal)
    fn = O.favor_causal if causal else O.favor_bidir
    got = fn(q[None, None], k[None, None], v[None, None], om[None], s)[0, 0]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


# -------------------------------------------------------------- feature maps
def test_positive_feature_hand_values():
    """phi_r(x) = m^-1/2 exp(omega_r.x - ||x||^2/2) on a non-symmetric omega:
    omega = [[1, 2], [-1, 0.5]], x = (0.5, -0.25): ||x||^2/2 = 0.15625,
    omega.x = (0.0, -0.625) -> phi = (exp(-0.15625), exp(-0.78125)) / sqrt(2)."""
    om = np.array([[1.0, 2.0], [-1.0, 0.5]])
    x = np.array([[0.5, -0.25]])
    got = O.feature_map_positive(x, om)
    want = np.array([[0.8553453273074225, 0.4578333617716143]]) / math.sqrt(2.0)
    np.testing.assert_allclose(got, want, rtol=1e-15)


def test_relu_feature_hand_values():
    """ReLU features with omega = I_d reduce to max(x, 0)/sqrt(d)."""
    x = np.array([[0.5, -0.25, 2.0, 0.0]])
    got = O.feature_map_relu(x, np.eye(4))
    np.testing.assert_allclose(got, [[0.25, 0.0, 1.0, 0.0]], rtol=0, atol=0)


def test_relu_attention_brute_force():
    rng = np.random.default_rng(3)
    L, d = 7, 5
    q, k, v = rng.normal(0, 1, (L, d)), rng.normal(0, 1, (L, d)), rng.normal(0, 1, (L, 2))
    om = rng.standard_normal((6, d))
    pq = np.maximum(q @ om.T, 0) / math.sqrt(6)
    pk = np.maximum(k @ om.T, 0) / math.sqrt(6)
    got = O.favor_bidir(q[None, None], k[None, None], v[None, None], om[None], 1.0, "relu")[0, 0]
    np.testing.assert_allclose(got, _brute(pq, pk, v, False), rtol=1e-12)


def test_relu_zero_denominator_gives_zero_row():
    """Disjoint supports make phi(q_1)^T phi(k_1) = 0: row 1 of causal output is 0."""
    pq = np.array([[1.0, 0.0], [1.0, 1.0]])
    pk = np.array([[0.0, 1.0], [1.0, 0.0]])
    v = np.array([[5.0], [7.0]])
    out = O.attn_from_features_causal(pq, pk, v)
    assert out[0, 0] == 0.0
    assert out[1, 0] == pytest.approx(6.0)


def test_omega_zero_closed_form():
    """omega = 0: phi(x) = m^-1/2 exp(-||x||^2/2) 1, so every bidirectional row
    equals sum_j e^{-||y_j||^2/2} v_j / sum_j e^{-||y_j||^2/2}."""
    rng = np.random.default_rng(8)
    L, d, m = 12, 3, 5
    q, k, v = rng.normal(0, 1, (L, d)), rng.normal(0, 1, (L, d)), rng.normal(0, 1, (L, 4))
    feats = O.feature_map_positive(k, np.zeros((m, d)))
    np.testing.assert_allclose(feats, np.exp(-0.5 * (k ** 2).sum(1))[:, None]
                               * np.ones((1, m)) / math.sqrt(m), rtol=1e-15)
    w = np.exp(-0.5 * (k ** 2).sum(1))
    want = (w @ v) / w.sum()
    got = O.favor_bidir(q[None, None], k[None, None], v[None, None], np.zeros((1, m, d)), 1.0)[0, 0]
    np.testing.assert_allclose(got, np.broadcast_to(want, got.shape), rtol=1e-12)


# --------------------------------------------------------- causal invariants
def test_causal_last_row_equals_bidirectional():
    """tril keeps the diagonal (Eq. 2), so the last causal row sees every key."""
    rng = np.random.default_rng(1)
    q, k, v = rng.normal(0, .5, (1, 2, 37, 8)), rng.normal(0, .5, (1, 2, 37, 8)), rng.normal(0, 1, (1, 2, 37, 5))
    om = np.stack([make_omega_orf(rng, 16, 8) for _ in range(2)])
    c = O.favor_causal(q, k, v, om, 0.6)
    b = O.favor_bidir(q, k, v, om, 0.6)
    np.testing.assert_allclose(c[..., -1, :], b[..., -1, :], rtol=1e-12)
    # L = 1: the only key is the query's own, output is v_1
    c1 = O.favor_causal(q[..., :1, :], k[..., :1, :], v[..., :1, :], om, 0.6)
    np.testing.assert_allclose(c1, v[..., :1, :], rtol=1e-14)


def test_causal_prefix_equals_rnn_and_block_size_free():
    rng = np.random.default_rng(2)
    L, m = 50, 6
    pq, pk = rng.uniform(0.01, 1, (L, m)), rng.uniform(0.01, 1, (L, m))
    v = rng.standard_normal((L, 3))
    ref = O.rnn_causal_from_features(pq, pk, v)
    for blk in (1, 7, 16, 512):
        np.testing.assert_allclose(O.attn_from_features_causal(pq, pk, v, block=blk), ref, rtol=1e-12)
    np.testing.assert_allclose(O.explicit_from_features(pq, pk, v, True), ref, rtol=1e-12)


# ------------------------------------------------------------------ invariants
def test_one_hot_values_give_attention_matrix():
    """[P] App. C.4: with V = I_L the output rows are the normalised attention
    matrix; rows sum to 1 and entries are non-negative for positive features."""
    rng = np.random.default_rng(4)
    L, d, m = 10, 4, 16
    q, k = rng.normal(0, .5, (L, d)), rng.normal(0, .5, (L, d))
    om = make_omega_orf(rng, m, d)
    pq, pk = O.feature_map_positive(q, om), O.feature_map_positive(k, om)
    for causal in (False, True):
        fn = O.attn_from_features_causal if causal else O.attn_from_features_bidir
        a = fn(pq, pk, np.eye(L))
        np.testing.assert_allclose(a.sum(1), 1.0, rtol=1e-13)
        assert (a >= 0).all()
        brute = _brute(pq, pk, np.eye(L), causal)
        np.testing.assert_allclose(a, brute, rtol=1e-12, atol=1e-15)
        if causal:
            assert np.all(np.triu(a, 1) == 0)


def test_constant_values_and_linearity_and_permutations():
    rng = np.random.default_rng(6)
    B, H, L, d, m = 1, 1, 20, 4, 8
    q, k = rng.normal(0, .5, (B, H, L, d)), rng.normal(0, .5, (B, H, L, d))
    om = make_omega_orf(rng, m, d)[None]
    const = np.broadcast_to(np.array([1.5, -2.0, 0.25]), (B, H, L, 3))
    np.testing.assert_allclose(O.favor_bidir(q, k, const, om, 1.0), const, rtol=1e-13)
    np.testing.assert_allclose(O.favor_causal(q, k, const, om, 1.0), const, rtol=1e-13)
    v = rng.normal(0, 1, (B, H, L, 3))
    base = O.favor_bidir(q, k, v, om, 1.0)
    np.testing.assert_allclose(O.favor_bidir(q, k, 3.0 * v, om, 1.0), 3.0 * base, rtol=1e-13)
    perm = rng.permutation(L)
    np.testing.assert_allclose(O.favor_bidir(q, k[..., perm, :], v[..., perm, :], om, 1.0), base, rtol=1e-12)
    fperm = rng.permutation(m)
    np.testing.assert_allclose(O.favor_bidir(q, k, v, om[:, fperm], 1.0), base, rtol=1e-12)


# ------------------------------------------------------- Monte Carlo (Lemma 1/2)
def test_lemma1_unbiased_and_lemma2_variance():
    """E[phi(x)^T phi(y)] = exp(x^T y) with iid Gaussian omega ([P] Lemma 1),
    and the single-feature variance matches Lemma 2's closed form
    MSE = (1/m) exp(||x+y||^2) SM(x,y)^2 (1 - exp(-||x+y||^2))."""
    rng = np.random.default_rng(12345)
    d = 6
    x = np.array([0.3, -0.2, 0.1, 0.4, 0.0, -0.1])
    y = np.array([-0.1, 0.25, 0.3, 0.2, -0.3, 0.05])
    sm = math.exp(x @ y)
    zz = float((x + y) @ (x + y))
    var1 = math.exp(zz) * sm ** 2 * (1 - math.exp(-zz))   # m = 1
    n = 400_000
    om = rng.standard_normal((n, d))
    est = O.feature_map_positive(x[None], om)[0] * O.feature_map_positive(y[None], om)[0] * n
    # each term n * phi_r(x) phi_r(y) is one m=1 sample of the estimator
    mean = est.mean()
    assert abs(mean - sm) < 5 * math.sqrt(var1 / n)
    assert est.var() == pytest.approx(var1, rel=0.03)
    # the m-feature estimator is the average of m single-feature samples
    m = 1000
    ests = (est[: (n // m) * m].reshape(-1, m).mean(1))
    assert ests.var() == pytest.approx(var1 / m, rel=0.25)


def _mean_exp_of_random_direction(z2, log_pdf, d):
    """E[exp(rho U.z)] with U uniform on S^{d-1} and rho of log-density log_pdf, by quadrature.

    E_U[exp(t U.e)] = Gamma(d/2) (t/2)^{1-d/2} I_{d/2-1}(t) (spherical mean of
    an exponential); scipy's exponentially scaled Bessel function keeps it finite.
    """
    special = pytest.importorskip("scipy.special")
    integrate = pytest.importorskip("scipy.integrate")
    zn = math.sqrt(z2)
    nu = d / 2 - 1

    def integrand(r):
        if r <= 0:
            return 0.0
        t = r * zn
        return math.exp(log_pdf(r) + math.lgamma(d / 2) + (1 - d / 2) * math.log(t / 2) + t) * special.ive(nu, t)

    val, _ = integrate.quad(integrand, 0, np.inf, limit=200)
    return val


def test_orthogonal_features_lower_mse_than_iid():
    """[P] Thm 2 / Thm 6: for m <= d orthogonal features have strictly smaller MSE
    than iid ones.  (The size of the gap is garbled on the page, so the test
    checks the direction, and the orthogonal MSE against its exact value: for
    an orthogonal pair with chi(d) lengths, omega_1 + omega_2 has a uniform
    direction and a chi(2d) length, which gives the pair covariance.)"""
    rng = np.random.default_rng(99)
    d = m = 8
    x = rng.normal(0, 0.35, d)
    y = rng.normal(0, 0.35, d)
    sm = math.exp(x @ y)
    reps = 20000
    e_iid = np.empty(reps)
    e_ort = np.empty(reps)
    for t in range(reps):
        oi = make_omega_iid(rng, m, d)
        oo = make_omega_orf(rng, m, d)
        e_iid[t] = O.feature_map_positive(x[None], oi)[0] @ O.feature_map_positive(y[None], oi)[0]
        e_ort[t] = O.feature_map_positive(x[None], oo)[0] @ O.feature_map_positive(y[None], oo)[0]
    mse_iid = np.mean((e_iid - sm) ** 2)
    mse_ort = np.mean((e_ort - sm) ** 2)
    zz = float((x + y) @ (x + y))
    mse_iid_closed = math.exp(zz) * sm ** 2 * (1 - math.exp(-zz)) / m
    assert mse_iid == pytest.approx(mse_iid_closed, rel=0.1)
    assert mse_ort < 0.9 * mse_iid
    lam2 = math.exp(-(x @ x) - (y @ y))
    def chi2d(r):      # log-density of a chi(2d) length
        return (2 * d - 1) * math.log(r) - r * r / 2 - (d - 1) * math.log(2) - math.lgamma(d)

    def chid_sqrt2(r):  # log-density of sqrt(2) * chi(d)
        return ((d - 1) * math.log(r / math.sqrt(2)) - r * r / 4 - (d / 2 - 1) * math.log(2)
                - math.lgamma(d / 2) - 0.5 * math.log(2))
    # quadrature sanity: a sqrt(2)*chi(d) length (iid pair sum) gives exp(||z||^2)
    assert _mean_exp_of_random_direction(zz, chid_sqrt2, d) == pytest.approx(math.exp(zz), rel=1e-8)
    cov_ort = lam2 * (_mean_exp_of_random_direction(zz, chi2d, d) - math.exp(zz))
    assert cov_ort < 0
    mse_ort_exact = mse_iid_closed + (1 - 1 / m) * cov_ort
    assert mse_ort == pytest.approx(mse_ort_exact, rel=0.1)
    # both estimators are unbiased
    assert abs(e_ort.mean() - sm) < 5 * math.sqrt(mse_ort / reps)


# --------------------------------------------------------------- exact softmax
def test_softmax_attention_matches_library_softmax():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(7)
    L, d = 30, 8
    q, k, v = rng.normal(0, 1, (L, d)), rng.normal(0, 1, (L, d)), rng.normal(0, 1, (L, 3))
    s = d ** -0.25
    w = scipy_special.softmax(q @ k.T / math.sqrt(d), axis=1)
    np.testing.assert_allclose(O.softmax_attention(q, k, v, s), w @ v, rtol=1e-12)
    logits = np.where(np.tril(np.ones((L, L), bool)), q @ k.T / math.sqrt(d), -np.inf)
    wc = scipy_special.softmax(logits, axis=1)
    np.testing.assert_allclose(O.softmax_attention(q, k, v, s, causal=True), wc @ v, rtol=1e-12)


def test_favor_converges_to_softmax_as_m_grows():
    """Performer §4.2 / Fig. 4 shape: output error vs exact softmax falls with m.

    Inputs use std 0.5 so ||x + y||^2 is about 2 and the Monte Carlo error is in
    its 1/m regime (Lemma 2: the relative variance per kernel entry grows like
    exp(||x + y||^2), so N(0,1) inputs need far larger m before it settles)."""
    rng = np.random.default_rng(21)
    L, d = 256, 16
    q, k, v = (rng.normal(0, 0.5, (L, d)) * d ** -0.25 for _ in range(3))
    exact = O.softmax_attention(q, k, v, 1.0)
    errs = []
    for m in (16, 256, 4096):
        e = []
        for _ in range(3):
            om = make_omega_orf(rng, m, d)
            got = O.favor_bidir(q[None, None], k[None, None], v[None, None], om[None], 1.0)[0, 0]
            e.append(np.mean((got - exact) ** 2))
        errs.append(np.mean(e))
    assert errs[0] > errs[1] > errs[2]
    assert errs[2] < errs[0] / 50


# ----------------------------------------------------------- generator pins
def test_orf_blocks_orthogonal_and_chi_lengths():
    rng = np.random.default_rng(0)
    d, m = 16, 48
    om = make_omega_orf(rng, m, d)
    assert om.shape == (m, d)
    for b in range(m // d):
        blk = om[b * d:(b + 1) * d]
        gram = blk @ blk.T
        np.testing.assert_allclose(gram, np.diag(np.diag(gram)), atol=1e-12)
    # row lengths are chi(d): E||w|| = sqrt(2) Gamma((d+1)/2)/Gamma(d/2), E||w||^2 = d
    lens = np.linalg.norm(np.concatenate([make_omega_orf(rng, 256, d) for _ in range(200)]), axis=1)
    mu1 = math.sqrt(2) * math.gamma((d + 1) / 2) / math.gamma(d / 2)
    assert lens.mean() == pytest.approx(mu1, rel=0.01)
    assert (lens ** 2).mean() == pytest.approx(d, rel=0.01)
    # marginally Gaussian: each coordinate ~ N(0, 1)
    allrows = np.concatenate([make_omega_orf(rng, 256, d) for _ in range(50)])
    assert allrows.std() == pytest.approx(1.0, rel=0.02)
    assert abs(allrows.mean()) < 0.02


def test_round_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    a = np.concatenate([rng.standard_normal(10000).astype(np.float32) * 10.0 ** rng.integers(-5, 5, 10000),
                        np.array([1.00390625, 1.01171875, -2.5, 0.0], np.float32)])
    want = torch.from_numpy(a).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(round_bf16(a), want)


def test_row_rel_err():
    ref = np.array([[1.0, -2.0], [0.0, 0.0]])
    got = np.array([[1.1, -2.0], [0.0, 0.5]])
    assert O.row_rel_err(got, ref) == pytest.approx(0.5)
    assert O.row_rel_err(got[:1], ref[:1]) == pytest.approx(0.05)


def test_elem_rel_err_hand_computed():
    """Element-wise measure with the 1%-of-row floor, values worked by hand.
    Row 0: max |o| = 2, floor 0.02.  Element 0: |1.1 - 1| / 1 = 0.1; element 1:
    |0.003 - 0.001| / max(0.001, 0.02) = 0.1; element 2: 0.  Row 1 (all-zero
    reference): absolute error 0.25.  Row 2: |0.5 - 0.4| / 0.4 = 0.25."""
    ref = np.array([[1.0, 0.001, -2.0], [0.0, 0.0, 0.0], [0.4, -0.1, 0.2]])
    got = np.array([[1.1, 0.003, -2.0], [0.0, 0.25, 0.0], [0.5, -0.1, 0.2]])
    assert O.elem_rel_err(got[:1], ref[:1]) == pytest.approx(0.1)
    assert O.elem_rel_err(got[1:2], ref[1:2]) == pytest.approx(0.25)
    assert O.elem_rel_err(got[2:], ref[2:]) == pytest.approx(0.25)
    assert O.elem_rel_err(got, ref) == pytest.approx(0.25)
    # the floor: an error of 1e-5 on an element of 1e-6 in a row of max 1 counts as 1e-5 / 1e-2
    assert O.elem_rel_err(np.array([[1.0, 1.1e-5]]), np.array([[1.0, 1e-6]])) == pytest.approx(1e-3)
    # a plain element-wise ratio where every element is above the floor
    assert O.elem_rel_err(np.array([[2.0, -3.3]]), np.array([[2.0, -3.0]])) == pytest.approx(0.1)
    assert O.elem_rel_err(np.zeros((0, 3)), np.zeros((0, 3))) == 0.0

