"""Pins for the oracle's backward (gradients of the forward attention).

The pages print no backward formulas, so the gradients are pinned to the
forward itself through routes that share none of the backward's algebra:
central finite differences of the (separately pinned) forward, the explicit
L x L form in which the output is linear in V, invariants of the normalised
attention, and special cases whose gradients are known in closed form.
"""
import numpy as np
import pytest

import oracle as O
from synth import make_omega_orf


def _inputs(seed, L=12, d=4, dv=3, m=8, std=0.6, H=1, B=1):
    rng = np.random.default_rng(seed)
    omega = np.stack([make_omega_orf(rng, m, d) for _ in range(H)])
    q = rng.normal(0, std, (B, H, L, d))
    k = rng.normal(0, std, (B, H, L, d))
    v = rng.normal(0, 1.0, (B, H, L, dv))
    g = rng.normal(0, 1.0, (B, H, L, dv))
    return omega, q, k, v, g


FWD = {"bidir": O.favor_bidir, "causal": O.favor_causal}
BWD = {"bidir": O.favor_bidir_backward, "causal": O.favor_causal_backward}


@pytest.mark.parametrize("mode", ["bidir", "causal"])
@pytest.mark.parametrize("kind", O.KINDS + ("softmax_hyp",))
def test_gradients_match_central_differences(mode, kind):
    """<grad, u> equals (f(x + h u) - f(x - h u)) / 2h for the loss <dO, out>,
    along random directions u of q, k and v (every element perturbed)."""
    omega, q, k, v, g = _inputs(1)
    s = 0.8
    grads = BWD[mode](q, k, v, g, omega, s, kind)
    rng = np.random.default_rng(7)
    h = 1e-6
    for which in range(3):
        for _ in range(3):
            u = rng.normal(size=(q, k, v)[which].shape)
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which] = args_p[which] + h * u
            args_m[which] = args_m[which] - h * u
            fp = np.sum(g * FWD[mode](*args_p, omega, s, kind))
            fm = np.sum(g * FWD[mode](*args_m, omega, s, kind))
            fd = (fp - fm) / (2 * h)
            an = np.sum(grads[which] * u)
            assert an == pytest.approx(fd, rel=2e-6, abs=1e-8), (which, an, fd)


@pytest.mark.parametrize("causal", [False, True])
def test_dv_equals_explicit_transpose(causal):
    """out = A V with A = D^-1 A_hat ([P] Eq. 1/2 with the kernel estimate), so
    dV = A^T dO exactly; A built by explicit loops over (i, j)."""
    omega, q, k, v, g = _inputs(2, L=9)
    s = 0.9
    pq = O.feature_map(s * q[0, 0], omega[0], "softmax_pos")
    pk = O.feature_map(s * k[0, 0], omega[0], "softmax_pos")
    L = pq.shape[0]
    a = np.zeros((L, L))
    for i in range(L):
        for j in range(L):
            if causal and j > i:
                continue
            a[i, j] = sum(pq[i, r] * pk[j, r] for r in range(pq.shape[1]))
        a[i] /= a[i].sum()
    dv_ref = a.T @ g[0, 0]
    fn = O.favor_causal_backward if causal else O.favor_bidir_backward
    _, _, dv = fn(q, k, v, g, omega, s)
    np.testing.assert_allclose(dv[0, 0], dv_ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("mode", ["bidir", "causal"])
def test_dv_columns_sum_to_upstream(mode):
    """Rows of the normalised attention sum to 1, so sum_j dV_j = sum_i dO_i."""
    omega, q, k, v, g = _inputs(3, L=40, d=8, dv=5, m=16)
    _, _, dv = BWD[mode](q, k, v, g, omega, 0.7)
    np.testing.assert_allclose(dv.sum(axis=2), g.sum(axis=2), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode", ["bidir", "causal"])
def test_query_key_grads_invariant_to_value_shift(mode):
    """out is a convex combination of value rows (positive features), so
    V -> V + 1 c^T shifts every output row by c and leaves the q and k
    gradients unchanged.  Dropping the denominator's term breaks this."""
    omega, q, k, v, g = _inputs(4, L=30, d=6, dv=4, m=12)
    c = np.array([3.0, -2.0, 0.5, 7.0])
    dq0, dk0, dv0 = BWD[mode](q, k, v, g, omega, 0.8)
    dq1, dk1, dv1 = BWD[mode](q, k, v + c, g, omega, 0.8)
    np.testing.assert_allclose(dq1, dq0, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk1, dk0, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv1, dv0, rtol=1e-12, atol=1e-13)


def test_zero_projection_gives_zero_query_gradient():
    """omega = 0: phi(x) = m^-1/2 exp(-||x||^2/2) 1, the same factor for every
    feature, so the bidirectional output does not depend on q and dq = 0;
    dk follows the closed form out = sum_j w_j v_j / sum_j w_j with
    w_j = exp(-s^2 ||k_j||^2 / 2):  dk_j = -s^2 k_j w_j (v_j - out) . dO_sum / W."""
    omega, q, k, v, g = _inputs(5, L=10)
    omega = np.zeros_like(omega)
    s = 0.7
    dq, dk, _ = O.favor_bidir_backward(q, k, v, g, omega, s)
    np.testing.assert_allclose(dq, 0.0, atol=1e-15)
    kk, vv, gs = k[0, 0], v[0, 0], g[0, 0].sum(axis=0)
    w = np.exp(-0.5 * s * s * np.sum(kk * kk, axis=1))
    out = (w @ vv) / w.sum()
    dk_ref = -(s * s) * kk * (w * ((vv - out) @ gs) / w.sum())[:, None]
    np.testing.assert_allclose(dk[0, 0], dk_ref, rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("kind", O.KINDS)
def test_causal_last_row_gradient_equals_bidirectional(kind):
    """Causal row L sees every key, as the bidirectional rows do ([P] Eq. 2 vs
    Eq. 1): with dO nonzero only on the last row, both backwards agree."""
    omega, q, k, v, g = _inputs(6, L=17)
    g[:, :, :-1] = 0.0
    a = O.favor_causal_backward(q, k, v, g, omega, 0.8, kind)
    ga = O.favor_bidir_backward(q, k, v, g, omega, 0.8, kind)
    np.testing.assert_allclose(a[0][:, :, -1], ga[0][:, :, -1], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(a[1], ga[1], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(a[2], ga[2], rtol=1e-11, atol=1e-13)
    np.testing.assert_array_equal(a[0][:, :, :-1], 0.0)


def test_causal_single_token():
    """L = 1: out_1 = v_1 whatever q and k (positive features), so dv = dO and
    dq = dk = 0."""
    omega, q, k, v, g = _inputs(7, L=1)
    dq, dk, dv = O.favor_causal_backward(q, k, v, g, omega, 0.9)
    np.testing.assert_allclose(dv, g, rtol=1e-14)
    np.testing.assert_allclose(dq, 0.0, atol=1e-14)
    np.testing.assert_allclose(dk, 0.0, atol=1e-14)


def test_causal_blocks_do_not_change_the_result():
    """The reverse sweep carries its suffix sums block by block: block sizes
    1, 5 and 512 give the same gradients (the same sums, regrouped)."""
    omega, q, k, v, g = _inputs(8, L=23)
    pq = O.feature_map(0.8 * q[0, 0], omega[0], "softmax_pos")
    pk = O.feature_map(0.8 * k[0, 0], omega[0], "softmax_pos")
    ref = O.attn_from_features_causal_vjp(pq, pk, v[0, 0], g[0, 0], block=512)
    for blk in (1, 5):
        got = O.attn_from_features_causal_vjp(pq, pk, v[0, 0], g[0, 0], block=blk)
        for a, b in zip(got, ref):
            np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-13)


def test_relu_zero_denominator_rows_have_zero_gradient():
    """ReLU features can give a causal row with den = 0 (its output is 0 by the
    convention); that row contributes nothing to any gradient."""
    d, m = 2, 2
    omega = np.eye(2)[None]                      # phi(x) = max(x, 0) / sqrt(2)
    q = np.array([[[[-1.0, -1.0], [1.0, 1.0], [1.0, 0.5]]]])
    k = np.array([[[[1.0, 1.0], [2.0, 1.0], [0.5, 1.0]]]])
    v = np.array([[[[1.0], [2.0], [3.0]]]])
    g = np.array([[[[5.0], [0.0], [0.0]]]])      # only row 1, whose den is 0
    dq, dk, dv = O.favor_causal_backward(q, k, v, g, omega, 1.0, "relu")
    assert O.favor_causal(q, k, v, omega, 1.0, "relu")[0, 0, 0, 0] == 0.0
    np.testing.assert_array_equal(dq, 0.0)
    np.testing.assert_array_equal(dk, 0.0)
    np.testing.assert_array_equal(dv, 0.0)


@pytest.mark.parametrize("mode", ["bidir", "causal"])
@pytest.mark.parametrize("kind", O.KINDS + ("softmax_hyp",))
def test_gradients_match_reverse_mode_autodiff(mode, kind):
    """Every element of dq, dk, dv against reverse-mode differentiation
    (PyTorch autograd, float64, CPU) of a forward written here from the
    definitions: the features of Lemma 1 (its first form, its hyperbolic
    second form with 2m features, or the ReLU map), the explicit
    L x L matrix A = phi(x) phi(y)^T (its lower triangle, diagonal included,
    for causal), out = A V / A 1.  Nothing is shared with the oracle."""
    torch = pytest.importorskip("torch")
    omega, q, k, v, g = _inputs(3)
    s = 0.8
    m = omega.shape[1]
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    om = torch.tensor(omega, dtype=torch.float64)

    def feat(x):
        proj = torch.einsum("bhld,hmd->bhlm", x, om)
        half = 0.5 * (x * x).sum(-1, keepdim=True)
        if kind == "softmax_pos":
            return torch.exp(proj - half) / m ** 0.5
        if kind == "softmax_hyp":
            return torch.cat([torch.exp(proj - half), torch.exp(-proj - half)], dim=-1) / (2 * m) ** 0.5
        return torch.relu(proj) / m ** 0.5

    A = torch.einsum("bhim,bhjm->bhij", feat(s * tq), feat(s * tk))
    if mode == "causal":
        A = torch.tril(A)
    den = A.sum(-1, keepdim=True)
    assert bool((den > 0).all())   # the seed gives no zero denominator (ReLU)
    ((A @ tv) / den * torch.tensor(g)).sum().backward()
    got = BWD[mode](q, k, v, g, omega, s, kind)
    for name, a, b in zip(("dq", "dk", "dv"), got, (tq.grad, tk.grad, tv.grad)):
        np.testing.assert_allclose(a, b.numpy(), rtol=1e-9, atol=1e-12, err_msg=name)


def _chunked_causal_feature_grads(pq, pk, v, g, chunk, per):
    """The causal gradients with respect to the features, evaluated chunk by
    chunk the way the tensor-core passes evaluate them: exclusive prefix
    states S, z of the keys before a chunk, exclusive suffix states T, t of
    the queries after it (T = sum phi_q dO^T / den, t = -sum phi_q go / den),
    carried across `per`-chunk pieces and rebuilt at each piece from the sums
    of the other pieces, and the masked products inside the chunk:
        den_i = phi_q,i . z + sum_{j<=i} A_ij,   A = Phi_Q Phi_K^T, C = dO V^T
        go_i  = (phi_q,i . (S dO_i) + sum_{j<=i} A_ij C_ij) / den_i
        dphi_q,i = (S dO_i - z go_i + sum_{j<=i} (C_ij - go_i) phi_k,j) / den_i
        dphi_k,j = T v_j + t + sum_{i>=j} (C_ij - go_i) phi_q,i / den_i
        dv_j     = T^T phi_k,j + sum_{i>=j} (phi_k,j . phi_q,i / den_i) dO_i"""
    L, m = pq.shape
    n_ch = -(-L // chunk)
    pieces = [list(range(p, min(n_ch, p + per))) for p in range(0, n_ch, per)]
    rows = lambda c: slice(c * chunk, min(L, (c + 1) * chunk))
    # key pieces -> exclusive prefix per piece
    tot = []
    for pc in pieces:
        S, z = np.zeros((m, v.shape[1])), np.zeros(m)
        for c in pc:
            S += pk[rows(c)].T @ v[rows(c)]
            z += pk[rows(c)].sum(0)
        tot.append((S, z))
    dpq, den_all, go_all = np.zeros_like(pq), np.zeros(L), np.zeros(L)
    for p, pc in enumerate(pieces):
        S = sum((t[0] for t in tot[:p]), np.zeros((m, v.shape[1])))
        z = sum((t[1] for t in tot[:p]), np.zeros(m))
        for c in pc:
            r = rows(c)
            n = r.stop - r.start
            Q, K, V, D = pq[r], pk[r], v[r], g[r]
            M = np.tril(np.ones((n, n)))
            A, Cm = Q @ K.T, D @ V.T
            den = Q @ z + (M * A).sum(1)
            go = ((Q * (D @ S.T)).sum(1) + (M * A * Cm).sum(1)) / den
            dpq[r] = (D @ S.T - np.outer(go, z) + (M * (Cm - go[:, None])) @ K) / den[:, None]
            den_all[r], go_all[r] = den, go
            S = S + K.T @ V
            z = z + K.sum(0)
    pqt = pq / den_all[:, None]
    tot = []
    for pc in pieces:
        T, t = np.zeros((m, v.shape[1])), np.zeros(m)
        for c in pc:
            T += pqt[rows(c)].T @ g[rows(c)]
            t -= (pqt[rows(c)] * go_all[rows(c), None]).sum(0)
        tot.append((T, t))
    dpk, dv = np.zeros_like(pk), np.zeros_like(v)
    for p, pc in enumerate(pieces):
        T = sum((x[0] for x in tot[p + 1:]), np.zeros((m, v.shape[1])))
        t = sum((x[1] for x in tot[p + 1:]), np.zeros(m))
        for c in reversed(pc):
            r = rows(c)
            n = r.stop - r.start
            Qt, K, V, D = pqt[r], pk[r], v[r], g[r]
            Mt = np.triu(np.ones((n, n)))
            W = Mt * (V @ D.T - go_all[r][None, :])
            dpk[r] = V @ T.T + t[None, :] + W @ Qt
            dv[r] = K @ T + (Mt * (K @ Qt.T)) @ D
            T = T + Qt.T @ D
            t = t - (Qt * go_all[r][:, None]).sum(0)
    return dpq, dpk, dv


@pytest.mark.parametrize("L,chunk,per", [(50, 8, 3), (64, 16, 1), (37, 8, 2)])
def test_causal_chunk_split_matches_the_derivative(L, chunk, per):
    """The chunked form of the causal gradients (prefix and suffix states of
    whole pieces, states carried across chunks inside a piece, masked
    products inside a chunk) gives the oracle's causal derivative on
    features, with ragged last chunks and keys whose features vanish (keys
    past the end of a tile)."""
    rng = np.random.default_rng(L)
    m, dv = 6, 3
    pq = rng.random((L, m)) + 0.05
    pk = rng.random((L, m)) + 0.05
    pk[-3:] = 0.0
    v = rng.normal(size=(L, dv))
    g = rng.normal(size=(L, dv))
    ref = O.attn_from_features_causal_vjp(pq, pk, v, g)
    got = _chunked_causal_feature_grads(pq, pk, v, g, chunk, per)
    for a, b in zip(got, ref):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)
