"""FAVOR+ attention (forward and its gradients) in plain float64 NumPy -- the oracle.

TEST INFRASTRUCTURE.  This module states, as directly as possible, what the
FAVOR+ forward path computes, and the exact derivative of it that the backward
path computes, so that the CUDA library can be checked against it.  It is slow on purpose: no blocking, fusion or reordering beyond what the
definitions below state, except that the causal prefix sum is carried block by
block so the [L, m, dv+1] prefix tensor is never held whole (the two are the
same sums).  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it; the library never does.

Sources (page title, then section / equation):
  [P]  Rethinking Attention with Performers (Choromanski et al.)
  [LA] Exploring Linear Attention: Does Attention Require a Softmax? (kexue)
  [EX] 040 . Performer explainer (wq-win.github.io)
  [PF] PermuteFormer: Efficient Relative Position Encoding for Long Sequences
  [RFA] Random Feature Attention (paperlayer summary of arXiv 2103.02143)

Readings taken where the pages are silent or garbled:
  * data scale s: x = s*q and y = s*k before the feature map ([P] §2.3 after
    Eq. 6: the sqrt(d) temperature is moved into the inputs; [EX] §1 uses
    s = d^-1/4).  V is never scaled.
  * no numerical stabiliser and no epsilon in the oracle (their values are
    lost on the page, [P] App. A.3/A.4); features are the plain definition.
  * a denominator that is exactly 0 (possible only for ReLU features) gives an
    output row of zeros.
  * causal attention includes the diagonal ([P] Eq. 2, tril keeps it).
  * two error measures.  Element-wise with a floor (the measure for fp32
    storage): max over elements of |g_ie - o_ie| / max(|o_ie|, 1e-2 max_e'|o_ie'|);
    the floor keeps the ratio defined where a signed output cancels to about
    zero.  Row-normwise (the measure for bf16 storage): max over rows i and
    columns e of |g_ie - o_ie| / max_e' |o_ie'|.

Every function takes float arrays of any float dtype and computes in float64.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "feature_map_positive", "feature_map_relu", "feature_map",
    "bidir_state", "attn_from_features_bidir", "attn_from_features_causal",
    "explicit_from_features", "rnn_causal_from_features",
    "favor_bidir", "favor_causal", "favor_feature_map",
    "favor_kv_state", "favor_attn_from_state", "favor_causal_from_state",
    "softmax_attention", "row_rel_err", "elem_rel_err", "KINDS",
    "feature_map_vjp", "attn_from_features_bidir_vjp", "attn_from_features_causal_vjp",
    "favor_bidir_backward", "favor_causal_backward",
    "feature_map_hyperbolic", "feature_map_trig", "VARIANT_KINDS", "n_features",
    "gated_causal_from_features", "favor_causal_gated", "permutation_power", "permute_features",
    "favor_permute",
]

KINDS = ("softmax_pos", "relu")
# Feature maps with l = 2 functions per projection row (Eq. 5): omega has M rows
# and the map has 2M features.
VARIANT_KINDS = ("softmax_hyp", "softmax_trig")


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def feature_map_positive(x, omega):
    """Positive random features of inputs x [..., d] (already scaled).

    [P] §2.3, Lemma 1 (Eq. 7) with h(x) = exp(-||x||^2/2), l = 1, f = exp in
    the general map of Eq. 5:  phi_r(x) = m^-1/2 * exp(omega_r . x - ||x||^2/2).
    [EX] §2 states the same per-feature formula.
    """
    x = _f64(x)
    omega = _f64(omega)
    m = omega.shape[0]
    proj = x @ omega.T
    sq = 0.5 * np.sum(x * x, axis=-1, keepdims=True)
    return np.exp(proj - sq) / np.sqrt(m)


def feature_map_relu(x, omega):
    """ReLU generalized-attention features: phi_r(x) = max(omega_r . x, 0) / sqrt(m).

    [P] §4.4 and App. A.4 (generalized attention with kernel = ReLU, i.e. f =
    ReLU, h = 1 in Eq. 5); [PF] §Performer uses phi(x) = max(x, 0) on the
    projected features.
    """
    x = _f64(x)
    omega = _f64(omega)
    m = omega.shape[0]
    return np.maximum(x @ omega.T, 0.0) / np.sqrt(m)


def feature_map_hyperbolic(x, omega):
    """Hyperbolic positive features SM^hyp+ ([P] Lemma 1, second form): Eq. 5 with
    h(x) = 2^-1/2 exp(-||x||^2/2), l = 2, f1(u) = exp(u), f2(u) = exp(-u):
        phi(x) = M^-1/2 h(x) (exp(omega_1.x), ..., exp(omega_M.x), exp(-omega_1.x), ..., exp(-omega_M.x))
    for the M rows of omega: 2M features.
    """
    x = _f64(x)
    omega = _f64(omega)
    M = omega.shape[0]
    proj = x @ omega.T
    sq = 0.5 * np.sum(x * x, axis=-1, keepdims=True)
    return np.concatenate([np.exp(proj - sq), np.exp(-proj - sq)], axis=-1) / np.sqrt(2.0 * M)


def feature_map_trig(x, omega):
    """Trigonometric features SM^trig ([P] §2.3 after Eq. 6): Eq. 5 with
    h(x) = exp(||x||^2/2), l = 2, f1 = sin, f2 = cos:
        phi(x) = M^-1/2 exp(||x||^2/2) (sin(omega_1.x), ..., sin(omega_M.x), cos(omega_1.x), ..., cos(omega_M.x))
    for the M rows of omega: 2M features, of either sign.
    """
    x = _f64(x)
    omega = _f64(omega)
    M = omega.shape[0]
    proj = x @ omega.T
    h = np.exp(0.5 * np.sum(x * x, axis=-1, keepdims=True))
    return h * np.concatenate([np.sin(proj), np.cos(proj)], axis=-1) / np.sqrt(M)


def n_features(kind, omega_rows):
    """Number of features of the map for ``omega_rows`` projection rows."""
    return 2 * omega_rows if kind in VARIANT_KINDS else omega_rows


def feature_map(x, omega, kind):
    if kind == "softmax_pos":
        return feature_map_positive(x, omega)
    if kind == "relu":
        return feature_map_relu(x, omega)
    if kind == "softmax_hyp":
        return feature_map_hyperbolic(x, omega)
    if kind == "softmax_trig":
        return feature_map_trig(x, omega)
    raise ValueError(f"unknown feature kind {kind!r}")


def _divide_rows(num, den):
    """out_i = num_i / den_i, and 0 where den_i == 0 exactly."""
    out = np.zeros_like(num)
    nz = den != 0.0
    out[nz] = num[nz] / den[nz, None]
    return out


def bidir_state(phi_k, v):
    """S = Phi_K^T V (m x dv) and z = Phi_K^T 1_L (m): the key/value summary of
    [EX] §2 (S = sum_j phi(k_j) v_j^T, z = sum_j phi(k_j)); together they are
    Buf1 = K'^T [V 1_L] of [P] App. B Alg. 1."""
    phi_k, v = _f64(phi_k), _f64(v)
    return phi_k.T @ v, phi_k.sum(axis=0)


def attn_from_features_bidir(phi_q, phi_k, v):
    """Bidirectional FAVOR attention from given features.

    [P] §2.2 Eq. 4 and App. B Alg. 1 (bidirectional branch):
        C = [V 1_L],  Buf1 = K'^T C  (m x (dv+1)),  Buf2 = Q' Buf1,
        split Buf2 = [Buf3 buf4] and return diag(buf4)^-1 Buf3.
    Equivalently S = Phi_K^T V, z = sum_j phi(k_j), out_i = phi(q_i)^T S /
    phi(q_i)^T z ([EX] §2).
    phi_q [Lq, m], phi_k [Lk, m], v [Lk, dv] -> out [Lq, dv].
    """
    phi_q, phi_k, v = _f64(phi_q), _f64(phi_k), _f64(v)
    c = np.concatenate([v, np.ones((v.shape[0], 1))], axis=1)
    buf1 = phi_k.T @ c
    buf2 = phi_q @ buf1
    return _divide_rows(buf2[:, :-1], buf2[:, -1])


def attn_from_features_causal(phi_q, phi_k, v, block=512):
    """Causal (unidirectional) FAVOR attention from given features.

    [P] App. B.1 Eq. 11: G_j = K'_j C_j^T, G^PS_i = sum_{j<=i} G_j, row i of
    tril(Q'K'^T) C equals G^PS_i^T Q'_i; then the same split/divide as Alg. 1.
    The prefix sum is carried across blocks of ``block`` rows: inside a block,
    sum_{j<=i} G_j = (state before the block) + sum over the block's rows
    j <= i, the latter written as tril(Q'_b K'_b^T) C_b.
    phi_q, phi_k [L, m], v [L, dv] -> out [L, dv].
    """
    phi_q, phi_k, v = _f64(phi_q), _f64(phi_k), _f64(v)
    L, m = phi_q.shape
    c = np.concatenate([v, np.ones((L, 1))], axis=1)
    state = np.zeros((m, c.shape[1]))
    buf2 = np.empty((L, c.shape[1]))
    for b0 in range(0, L, block):
        b1 = min(L, b0 + block)
        pq, pk, cb = phi_q[b0:b1], phi_k[b0:b1], c[b0:b1]
        buf2[b0:b1] = np.tril(pq @ pk.T) @ cb + pq @ state
        state = state + pk.T @ cb
    return _divide_rows(buf2[:, :-1], buf2[:, -1])


def explicit_from_features(phi_q, phi_k, v, causal):
    """The L x L form: A_hat = Q' K'^T (masked by tril if causal), D^-1 A_hat V.

    [P] Eq. 1/2 with A replaced by the kernel estimate of Eq. 3-4; only for
    small L (it builds the L x L matrix the method avoids).
    """
    a = _f64(phi_q) @ _f64(phi_k).T
    if causal:
        a = np.tril(a)
    return _divide_rows(a @ _f64(v), a.sum(axis=1))


def rnn_causal_from_features(phi_q, phi_k, v):
    """Token-by-token recurrence S_t = S_{t-1} + phi(k_t) v_t^T, z_t = z_{t-1} + phi(k_t),
    out_t = phi(q_t)^T S_t / phi(q_t)^T z_t ([LA] "Autoregressive Generation";
    [RFA] causal RFA).  A pure-Python loop: small L only."""
    phi_q, phi_k, v = _f64(phi_q), _f64(phi_k), _f64(v)
    L, m = phi_q.shape
    s = np.zeros((m, v.shape[1]))
    z = np.zeros(m)
    out = np.zeros((L, v.shape[1]))
    for t in range(L):
        s += np.outer(phi_k[t], v[t])
        z += phi_k[t]
        den = phi_q[t] @ z
        out[t] = (phi_q[t] @ s) / den if den != 0.0 else 0.0
    return out


def _per_head(q, k, v, omega, data_scale, kind, fn):
    q, k, v = _f64(q), _f64(k), _f64(v)
    omega = _f64(omega)
    B, H, L, _ = q.shape
    out = np.empty((B, H, L, v.shape[-1]))
    for b in range(B):
        for h in range(H):
            pq = feature_map(data_scale * q[b, h], omega[h], kind)
            pk = feature_map(data_scale * k[b, h], omega[h], kind)
            out[b, h] = fn(pq, pk, v[b, h])
    return out


def favor_bidir(q, k, v, omega, data_scale, kind="softmax_pos"):
    """FAVOR+ bidirectional forward on [B,H,L,d] inputs with omega [H,m,d]."""
    return _per_head(q, k, v, omega, data_scale, kind, attn_from_features_bidir)


def favor_causal(q, k, v, omega, data_scale, kind="softmax_pos"):
    """FAVOR+ causal forward on [B,H,L,d] inputs with omega [H,m,d]."""
    return _per_head(q, k, v, omega, data_scale, kind, attn_from_features_causal)


def favor_feature_map(x, omega, data_scale, kind="softmax_pos"):
    """phi(s*x) for x [B,H,L,d], omega [H,m,d] -> [B,H,L,m]."""
    x = _f64(x)
    omega = _f64(omega)
    B, H, L, _ = x.shape
    out = np.empty((B, H, L, n_features(kind, omega.shape[1])))
    for h in range(H):
        out[:, h] = feature_map(data_scale * x[:, h], omega[h], kind)
    return out


def favor_kv_state(k, v, omega, data_scale, kind="softmax_pos"):
    """Key/value state of [B,H,L,*] keys and values: state[b,h] = K'^T [V 1_L]
    ([P] App. B Alg. 1, Buf1), i.e. columns 0..dv-1 hold S = sum_j phi(k_j) v_j^T
    and column dv holds z = sum_j phi(k_j) ([EX] §2).  -> [B,H,m,dv+1]."""
    k, v, omega = _f64(k), _f64(v), _f64(omega)
    B, H, L, _ = k.shape
    m, dv = n_features(kind, omega.shape[1]), v.shape[-1]
    out = np.empty((B, H, m, dv + 1))
    for b in range(B):
        for h in range(H):
            pk = feature_map(data_scale * k[b, h], omega[h], kind)
            out[b, h] = pk.T @ np.concatenate([v[b, h], np.ones((L, 1))], axis=1)
    return out


def favor_attn_from_state(q, state, omega, data_scale, kind="softmax_pos"):
    """Readout against a given state ([P] App. B Alg. 1: Buf2 = Q' Buf1, split,
    divide): out_i = phi(q_i)^T S / phi(q_i)^T z for every query of [B,H,Lq,d];
    the keys behind the state may be another sequence (cross attention)."""
    q, state, omega = _f64(q), _f64(state), _f64(omega)
    B, H, Lq, _ = q.shape
    out = np.empty((B, H, Lq, state.shape[-1] - 1))
    for b in range(B):
        for h in range(H):
            buf2 = feature_map(data_scale * q[b, h], omega[h], kind) @ state[b, h]
            out[b, h] = _divide_rows(buf2[:, :-1], buf2[:, -1])
    return out


def favor_causal_from_state(q, k, v, state, omega, data_scale, kind="softmax_pos"):
    """Causal attention over T new tokens that follow the keys summarised by
    ``state`` ([P] App. B.1 Eq. 11 with the prefix sum started at ``state``
    instead of 0; the RNN form of [LA] "Autoregressive Generation" / [RFA]):
    out_i = phi(q_i)^T (S + sum_{j<=i} phi(k_j) v_j^T) / phi(q_i)^T (z + sum_{j<=i} phi(k_j)).
    Returns (out [B,H,T,dv], new state = state + K'^T [V 1])."""
    q, k, v, state, omega = _f64(q), _f64(k), _f64(v), _f64(state), _f64(omega)
    B, H, T, _ = q.shape
    out = np.empty((B, H, T, v.shape[-1]))
    new = np.empty_like(state)
    for b in range(B):
        for h in range(H):
            pq = feature_map(data_scale * q[b, h], omega[h], kind)
            pk = feature_map(data_scale * k[b, h], omega[h], kind)
            c = np.concatenate([v[b, h], np.ones((T, 1))], axis=1)
            buf2 = np.tril(pq @ pk.T) @ c + pq @ state[b, h]
            out[b, h] = _divide_rows(buf2[:, :-1], buf2[:, -1])
            new[b, h] = state[b, h] + pk.T @ c
    return out, new


# ----------------------------------------------------------------- backward
# The pages time the backward pass ([P] §4.1, Fig. 3) but print no formulas for
# it, so the backward below is the exact reverse-mode derivative of the forward
# steps above, taken step by step in reverse order.  For a scalar loss with
# upstream gradient dO = d loss / d out:
#   out_i = Buf3_i / buf4_i        ->  dBuf3_i = dO_i / buf4_i,
#                                      dbuf4_i = -(dO_i . out_i) / buf4_i
#   (a row with buf4_i == 0 has out_i = 0, a constant: both are 0 there)
#   Buf2 = Q' Buf1                 ->  dQ' = dBuf2 Buf1^T,  dBuf1 = Q'^T dBuf2
#   Buf1 = K'^T C, C = [V 1]       ->  dK' = C dBuf1^T,     dC = K' dBuf1
# and the feature maps' own derivatives (feature_map_vjp).

def feature_map_vjp(x, omega, kind, dphi):
    """d loss / d x for phi = feature_map(x, omega, kind), given dphi = d loss / d phi.

    Positive features ([P] Lemma 1): d phi_r / d x = phi_r (omega_r - x), so
        dx = (dphi * phi) Omega - x * sum_r (dphi * phi)_r.
    ReLU features ([P] App. A.4): d phi_r / d x = m^-1/2 [omega_r . x > 0] omega_r
    (the derivative of max(u, 0) is taken as 0 at u = 0).
    x [n, d], omega [m, d], dphi [n, m] -> [n, d].
    """
    x, omega, dphi = _f64(x), _f64(omega), _f64(dphi)
    if kind == "softmax_pos":
        g = dphi * feature_map_positive(x, omega)
        return g @ omega - x * g.sum(axis=1, keepdims=True)
    if kind == "relu":
        mask = (x @ omega.T) > 0.0
        return (np.where(mask, dphi, 0.0) @ omega) / np.sqrt(omega.shape[0])
    if kind == "softmax_hyp":
        # phi_r = (2M)^-1/2 exp(+-omega_r . x - ||x||^2/2): d phi_r / d x = phi_r (+-omega_r - x)
        g = dphi * feature_map_hyperbolic(x, omega)
        M = omega.shape[0]
        return g[:, :M] @ omega - g[:, M:] @ omega - x * g.sum(axis=1, keepdims=True)
    raise ValueError(f"no derivative for feature kind {kind!r}")


def _dbuf2(buf2, dout):
    """[dBuf3 dbuf4] from Buf2 = [Buf3 buf4] and dO (rows with buf4 == 0 give 0)."""
    num, den = buf2[:, :-1], buf2[:, -1]
    out = _divide_rows(num, den)
    d = np.zeros_like(buf2)
    nz = den != 0.0
    d[nz, :-1] = dout[nz] / den[nz, None]
    d[nz, -1] = -np.sum(dout[nz] * out[nz], axis=1) / den[nz]
    return d


def attn_from_features_bidir_vjp(phi_q, phi_k, v, dout):
    """Gradients of attn_from_features_bidir with respect to its three inputs.

    Reverse of [P] App. B Alg. 1 (bidirectional branch), see the table above.
    Returns (dphi_q [Lq, m], dphi_k [Lk, m], dv [Lk, dv]).
    """
    phi_q, phi_k, v, dout = _f64(phi_q), _f64(phi_k), _f64(v), _f64(dout)
    c = np.concatenate([v, np.ones((v.shape[0], 1))], axis=1)
    buf1 = phi_k.T @ c
    d2 = _dbuf2(phi_q @ buf1, dout)
    dbuf1 = phi_q.T @ d2
    return d2 @ buf1.T, c @ dbuf1.T, (phi_k @ dbuf1)[:, :-1]


def attn_from_features_causal_vjp(phi_q, phi_k, v, dout, block=512):
    """Gradients of attn_from_features_causal with respect to its three inputs.

    Reverse of [P] App. B.1 Eq. 11.  With G^PS_i = sum_{j<=i} K'_j C_j^T (the
    forward prefix sums) and H_j = sum_{i>=j} Q'_i dBuf2_i^T (suffix sums of
    the reverse pass):
        dQ'_i = G^PS_i dBuf2_i,   dK'_j = H_j C_j,   dC_j = H_j^T K'_j.
    Both sums are carried across blocks of ``block`` rows as in the forward:
    the prefix from the first block on, the suffix from the last block back;
    inside a block the within-block terms are written with tril of the
    block's row-by-row products.
    """
    phi_q, phi_k, v, dout = _f64(phi_q), _f64(phi_k), _f64(v), _f64(dout)
    L, m = phi_q.shape
    c = np.concatenate([v, np.ones((L, 1))], axis=1)
    # forward sweep: Buf2 (for dBuf2) and dQ' from the prefix sums
    g_ps = np.zeros((m, c.shape[1]))
    d2 = np.empty((L, c.shape[1]))
    dphi_q = np.empty((L, m))
    for b0 in range(0, L, block):
        b1 = min(L, b0 + block)
        pq, pk, cb = phi_q[b0:b1], phi_k[b0:b1], c[b0:b1]
        d2[b0:b1] = _dbuf2(np.tril(pq @ pk.T) @ cb + pq @ g_ps, dout[b0:b1])
        dphi_q[b0:b1] = np.tril(d2[b0:b1] @ cb.T) @ pk + d2[b0:b1] @ g_ps.T
        g_ps = g_ps + pk.T @ cb
    # reverse sweep: dK' and dC from the suffix sums
    h_s = np.zeros((m, c.shape[1]))
    dphi_k = np.empty((L, m))
    dc = np.empty_like(c)
    starts = list(range(0, L, block))
    for b0 in reversed(starts):
        b1 = min(L, b0 + block)
        pq, pk, cb, db = phi_q[b0:b1], phi_k[b0:b1], c[b0:b1], d2[b0:b1]
        dphi_k[b0:b1] = np.tril(db @ cb.T).T @ pq + cb @ h_s.T
        dc[b0:b1] = np.tril(pq @ pk.T).T @ db + pk @ h_s
        h_s = h_s + pq.T @ db
    return dphi_q, dphi_k, dc[:, :-1]


def _per_head_backward(q, k, v, dout, omega, data_scale, kind, vjp):
    q, k, v, dout, omega = _f64(q), _f64(k), _f64(v), _f64(dout), _f64(omega)
    dq, dk, dvv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    B, H = q.shape[:2]
    for b in range(B):
        for h in range(H):
            x, y = data_scale * q[b, h], data_scale * k[b, h]
            pq, pk = feature_map(x, omega[h], kind), feature_map(y, omega[h], kind)
            dpq, dpk, dvv[b, h] = vjp(pq, pk, v[b, h], dout[b, h])
            dq[b, h] = data_scale * feature_map_vjp(x, omega[h], kind, dpq)
            dk[b, h] = data_scale * feature_map_vjp(y, omega[h], kind, dpk)
    return dq, dk, dvv


def favor_bidir_backward(q, k, v, dout, omega, data_scale, kind="softmax_pos"):
    """(dq, dk, dv) of favor_bidir for the upstream gradient dout [B,H,L,dv]."""
    return _per_head_backward(q, k, v, dout, omega, data_scale, kind, attn_from_features_bidir_vjp)


def favor_causal_backward(q, k, v, dout, omega, data_scale, kind="softmax_pos"):
    """(dq, dk, dv) of favor_causal for the upstream gradient dout [B,H,L,dv]."""
    return _per_head_backward(q, k, v, dout, omega, data_scale, kind, attn_from_features_causal_vjp)


# ------------------------------------------------------------ gated causal (RFA-Gate)
def gated_causal_from_features(phi_q, phi_k, v, gate):
    """Causal attention with a gated (decaying) state, token by token.

    [RFA] §3.2 RFA-GATE: scalar gates g_t in [0, 1], computed by the model from
    the timestep's input, decay the history of both the value state and the
    normalisation state.  Reading taken (the page states the gate only in
    words): the gate interpolates between the history and the current token,
        S_t = g_t S_{t-1} + (1 - g_t) phi(k_t) v_t^T,
        z_t = g_t z_{t-1} + (1 - g_t) phi(k_t),
        out_t = phi(q_t)^T S_t / phi(q_t)^T z_t   (0 if the denominator is 0),
    with S_0 = 0, z_0 = 0 as in [RFA] A.3.  A pure-Python loop over t.
    phi_q, phi_k [L, m], v [L, dv], gate [L] -> out [L, dv].
    """
    phi_q, phi_k, v, gate = _f64(phi_q), _f64(phi_k), _f64(v), _f64(gate)
    L, m = phi_q.shape
    s = np.zeros((m, v.shape[1]))
    z = np.zeros(m)
    out = np.zeros((L, v.shape[1]))
    for t in range(L):
        g = gate[t]
        s = g * s + (1.0 - g) * np.outer(phi_k[t], v[t])
        z = g * z + (1.0 - g) * phi_k[t]
        den = phi_q[t] @ z
        out[t] = (phi_q[t] @ s) / den if den != 0.0 else 0.0
    return out


def favor_causal_gated(q, k, v, gate, omega, data_scale, kind="softmax_pos"):
    """RFA-Gate causal attention on [B,H,L,*] inputs with gates [B,H,L]."""
    q, k, v, gate, omega = _f64(q), _f64(k), _f64(v), _f64(gate), _f64(omega)
    B, H, L, _ = q.shape
    out = np.empty((B, H, L, v.shape[-1]))
    for b in range(B):
        for h in range(H):
            pq = feature_map(data_scale * q[b, h], omega[h], kind)
            pk = feature_map(data_scale * k[b, h], omega[h], kind)
            out[b, h] = gated_causal_from_features(pq, pk, v[b, h], gate[b, h])
    return out


# ------------------------------------------------------------ PermuteFormer
def permutation_power(perm, i):
    """pi^i as an index array: pi^i(a) = pi(pi(...pi(a))) (i times); pi^0 = identity.
    [PF] §Computational cost: powers of a permutation are permutations, composed
    by indexing."""
    perm = np.asarray(perm)
    out = np.arange(len(perm))
    for _ in range(i):
        out = perm[out]
    return out


def permute_features(phi, perm, r, sign):
    """Position-dependent transform of PermuteFormer ([PF] §PermuteFormer, the
    solution chosen for Eq. 9-10): row i of phi [L, m] becomes
    r^(sign*i) P_pi^i phi_i, where P_pi has P_ab = 1 iff pi(a) = b, so
    (P_pi^i phi)_a = phi_{pi^i(a)} (a gather by pi^i).  Queries take sign = +1
    and keys sign = -1, so that the similarity of query i and key j is
    r^(i-j) phi(q_i)^T P_pi^(j-i) phi(k_j): it depends on i - j only.
    Positions i count from 0 (only differences matter)."""
    phi = _f64(phi)
    out = np.empty_like(phi)
    idx = np.arange(phi.shape[1])
    perm = np.asarray(perm)
    for i in range(phi.shape[0]):
        out[i] = (float(r) ** (sign * i)) * phi[i, idx]
        idx = perm[idx]           # pi^(i+1)
    return out


def favor_permute(q, k, v, omega, data_scale, perm, r, causal, kind="softmax_pos"):
    """PermuteFormer attention ([PF] §PermuteFormer): Performer features of q
    and k, transformed by permute_features (r applies to causal attention; the
    page takes r = 1 for bidirectional models), then the usual bidirectional
    (Alg. 1) or causal (Eq. 11) attention from features.  perm [H, m] holds one
    permutation of the feature indices per head, r [H] one decay per head."""
    q, k, v, omega = _f64(q), _f64(k), _f64(v), _f64(omega)
    B, H, L, _ = q.shape
    out = np.empty((B, H, L, v.shape[-1]))
    for b in range(B):
        for h in range(H):
            rr = float(r[h]) if causal else 1.0
            pq = permute_features(feature_map(data_scale * q[b, h], omega[h], kind), perm[h], rr, +1)
            pk = permute_features(feature_map(data_scale * k[b, h], omega[h], kind), perm[h], rr, -1)
            fn = attn_from_features_causal if causal else attn_from_features_bidir
            out[b, h] = fn(pq, pk, v[b, h])
    return out


def softmax_attention(q, k, v, data_scale, causal=False):
    """Exact softmax attention of [P] Eq. 1 (bidirectional) / Eq. 2 (causal) with
    A = exp(x_i . y_j), x = s*q, y = s*k (s = d^-1/4 gives q.k/sqrt(d)).

    Each row is shifted by its max before exp; the shift cancels in D^-1 A V.
    Inputs [L, d] / [L, dv] (one head) or [B,H,L,*] (looped).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim == 4:
        out = np.empty(q.shape[:3] + (v.shape[-1],))
        for b in range(q.shape[0]):
            for h in range(q.shape[1]):
                out[b, h] = softmax_attention(q[b, h], k[b, h], v[b, h], data_scale, causal)
        return out
    logits = (data_scale * q) @ (data_scale * k).T
    if causal:
        mask = np.tril(np.ones(logits.shape, dtype=bool))
        logits = np.where(mask, logits, -np.inf)
    logits = logits - logits.max(axis=1, keepdims=True)
    a = np.exp(logits)
    return (a @ v) / a.sum(axis=1, keepdims=True)


def row_rel_err(got, ref):
    """max_{rows i, cols e} |got_ie - ref_ie| / max_e' |ref_ie'| over the last axis.

    Rows whose reference is all zeros use an absolute error instead.
    """
    got = _f64(got)
    ref = _f64(ref)
    scale = np.max(np.abs(ref), axis=-1, keepdims=True)
    scale = np.where(scale > 0, scale, 1.0)
    return float(np.max(np.abs(got - ref) / scale)) if ref.size else 0.0


def elem_rel_err(got, ref, floor=1e-2):
    """max over elements of |got_ie - ref_ie| / max(|ref_ie|, floor * max_e' |ref_ie'|).

    The element-wise relative error, with each element's divisor held at least
    at `floor` times the largest magnitude of its row (last axis), so that
    entries of a signed output that cancel to about zero do not make the ratio
    unbounded.  Rows whose reference is all zeros use an absolute error.
    """
    got = _f64(got)
    ref = _f64(ref)
    if not ref.size:
        return 0.0
    rmax = np.max(np.abs(ref), axis=-1, keepdims=True)
    scale = np.maximum(np.abs(ref), floor * rmax)
    scale = np.where(scale > 0, scale, 1.0)
    return float(np.max(np.abs(got - ref) / scale))
