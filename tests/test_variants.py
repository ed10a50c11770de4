"""GPU parity of the feature-map variants against the float64 oracle:
hyperbolic positive features (tensor-core and CUDA-core shapes, forward,
stateful calls and backward), trigonometric features (tensor-core and
CUDA-core shapes, forward and stateful calls) and SMREG projections
(regularized omega rows)."""
import numpy as np
import pytest

import oracle as O
import random_feature_gb300 as R
from synth import CONFIGS, make_upstream_grad, make_workload

from _util import TOL, to_dev, to_host

pytestmark = pytest.mark.gpu

SHAPES = [
    ("d64_m256_bf16", "bidir_bf16", dict(B=2, H=2)),        # tensor-core shape (hyp runs there)
    ("d32_m64_bf16", "bidir_bf16", dict(B=1, H=3, d=32, dv=16, m=64)),
    ("d16_m64_f32", "approx_f32", dict(B=2, H=2, m=64, dv=32)),
]


def trig_row_condition(q, k, v, omega, s, causal):
    """Per output row i: (max_e |Phi_q| |S|[i, e] + max|out_i| (|Phi_q| |z|)_i) / (|den_i| max|out_i|),
    the factor by which rounding of the sums in num_i and den_i is amplified in
    out_i relative to its row.  Near 1 for positive features; large for
    trigonometric ones, whose mixed-sign terms cancel (the §2.3 instability)."""
    kind = "softmax_trig"
    B, H, L, _ = q.shape
    Lk = k.shape[2]   # the keys may be another sequence (attention from a state)
    cond = np.empty((B, H, L))
    for b in range(B):
        for h in range(H):
            pq = O.feature_map(s * q[b, h], omega[h], kind)
            pk = O.feature_map(s * k[b, h], omega[h], kind)
            c = np.concatenate([v[b, h], np.ones((Lk, 1))], axis=1)
            if causal:
                g = np.cumsum(pk[:, :, None] * c[:, None, :], axis=0)           # [L, m, dv+1]
                ga = np.cumsum(np.abs(pk)[:, :, None] * np.abs(c)[:, None, :], axis=0)
                num = np.einsum("lr,lre->le", pq, g)
                anum = np.einsum("lr,lre->le", np.abs(pq), ga)
            else:
                num = pq @ (pk.T @ c)
                anum = np.abs(pq) @ (np.abs(pk).T @ np.abs(c))
            den = num[:, -1]
            out = num[:, :-1] / den[:, None]
            rm = np.abs(out).max(axis=1)
            cond[b, h] = (anum[:, :-1].max(axis=1) + rm * anum[:, -1]) / (np.abs(den) * rm)
    return cond


# Unit roundoff of the arithmetic whose errors a trigonometric row's condition
# amplifies: fp32 sums on the CUDA cores; on the tensor-core shape the features,
# the state image and the masked products are bf16 operands.
TRIG_UNIT = {"f32": 2.0 ** -24, "bf16": 2.0 ** -9}


def assert_trig_rows(out, ref, cond, dtype):
    """Row by row: the dtype's stated tolerance plus 4 unit roundoffs times the
    row's condition (mixed-sign cancellation, the instability of Rethinking
    Attention with Performers §2.3, amplifies rounding by that factor)."""
    scale = np.maximum(np.abs(ref).max(axis=-1), 1e-300)
    err = np.abs(out - ref).max(axis=-1) / scale
    bound = TOL[dtype] + 4 * TRIG_UNIT[dtype] * cond
    assert np.all(err <= bound), float(np.max(err / bound))


def _setup(shape, kind, L, seed, **extra):
    _, base, over = shape
    w = CONFIGS[base].replace(L=L, **over, **extra)
    omega, q, k, v = make_workload(w, seed)
    if kind in O.VARIANT_KINDS:
        omega = np.ascontiguousarray(omega[:, : w.m // 2])
    f = R.Favor(w.H, w.m, w.d, w.dv, kind, w.dtype, omega, w.data_scale, w.B, w.L)
    return w, omega, q, k, v, f


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("kind", O.VARIANT_KINDS)
@pytest.mark.parametrize("mode", ["bidir", "causal"])
def test_variant_attention(shape, kind, mode):
    w, omega, q, k, v, f = _setup(shape, kind, 1100, 51)
    with f:
        out = to_host(f.attn(*(to_dev(a, w.dtype) for a in (q, k, v)), causal=(mode == "causal")))
        assert R.favor_device_error(f.handle) == 0
    ref = (O.favor_causal if mode == "causal" else O.favor_bidir)(q, k, v, omega, w.data_scale, kind)
    assert np.isfinite(out).all()
    if kind == "softmax_trig":
        cond = trig_row_condition(q, k, v, omega, w.data_scale, mode == "causal")
        assert_trig_rows(out, ref, cond, w.dtype)
    else:
        assert O.row_rel_err(out, ref) <= TOL[w.dtype]


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("kind", O.VARIANT_KINDS)
def test_variant_feature_map(shape, kind):
    w, omega, q, k, v, f = _setup(shape, kind, 300, 52)
    with f:
        phi = to_host(f.feature_map(to_dev(q, w.dtype)))
    ref = O.favor_feature_map(q, omega, w.data_scale, kind)
    assert phi.shape == ref.shape
    tol = 1e-5 if w.dtype == "f32" else 1e-2
    np.testing.assert_allclose(phi, ref, rtol=tol, atol=tol * np.abs(ref).max())


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("kind", O.VARIANT_KINDS)
def test_variant_stateful_calls(shape, kind):
    """Key/value state, cross attention from it, and causal steps continuing it."""
    w, omega, q, k, v, f = _setup(shape, kind, 700, 53)
    with f:
        kd, vd = to_dev(k, w.dtype), to_dev(v, w.dtype)
        st = f.kv_state(kd, vd)
        ref_st = O.favor_kv_state(k, v, omega, w.data_scale, kind)
        if kind == "softmax_hyp":   # the positive kind's per-head key shift, on the mirrored rows
            sq = np.max(np.sum(np.asarray(omega, np.float64) ** 2, axis=-1), axis=-1)
            ref_st = ref_st * np.exp(-np.maximum(0.0, 0.5 * sq - 60.0))[None, :, None, None]
        got_st = to_host(st)
        assert O.row_rel_err(got_st.reshape(-1, w.dv + 1), ref_st.reshape(-1, w.dv + 1)) <= TOL[w.dtype]
        q2 = q[:, :, :300]
        out = to_host(f.attn_from_state(to_dev(q2, w.dtype), st))
        ref = O.favor_attn_from_state(q2, ref_st, omega, w.data_scale, kind)
        if kind == "softmax_trig":
            assert_trig_rows(out, ref, trig_row_condition(q2, k, v, omega, w.data_scale, False), w.dtype)
        else:
            assert O.row_rel_err(out, ref) <= TOL[w.dtype]
        # 5 causal steps of one token each after the 700-token state
        _, qn, kn, vn = make_workload(w.replace(L=5), 54)
        outs = []
        for t in range(5):
            sl = slice(t, t + 1)
            outs.append(to_host(f.causal_step(*(to_dev(a[:, :, sl], w.dtype) for a in (qn, kn, vn)), st)))
        ref_out, _ = O.favor_causal_from_state(qn, kn, vn, ref_st, omega, w.data_scale, kind)
        assert O.row_rel_err(np.concatenate(outs, axis=2), ref_out) <= TOL[w.dtype]


@pytest.mark.parametrize("shape", SHAPES[::2], ids=[s[0] for s in SHAPES[::2]])
@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_hyperbolic_backward(shape, causal):
    w, omega, q, k, v, f = _setup(shape, "softmax_hyp", 700, 55)
    g = make_upstream_grad(w, 55)
    ref = (O.favor_causal_backward if causal else O.favor_bidir_backward)(q, k, v, g, omega, w.data_scale,
                                                                          "softmax_hyp")
    with f:
        got = [to_host(t) for t in f.attn_backward(*(to_dev(a, w.dtype) for a in (q, k, v, g)), causal=causal)]
    from test_backward import TOL_GRAD, grad_err
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        assert grad_err(a, b) <= TOL_GRAD[w.dtype], name


def test_trig_backward_and_noalloc_are_unsupported():
    w, omega, q, k, v, f = _setup(SHAPES[2], "softmax_trig", 64, 56)
    with f:
        dev = [to_dev(a, w.dtype) for a in (q, k, v, v)]
        with pytest.raises(R.FavorError) as ei:
            f.attn_backward(*dev)
        assert ei.value.status == R.FAVOR_ERR_UNSUPPORTED
    import torch
    om = torch.zeros((w.H, w.m, w.d), device="cuda")
    out = torch.empty_like(dev[2])
    with pytest.raises(R.FavorError) as ei:
        R.favor_attn_bidir_noalloc(om, w.H, w.m, w.d, w.dv, "softmax_trig", w.dtype, w.data_scale,
                                   dev[0], dev[1], dev[2], out, w.B, w.L)
    assert ei.value.status == R.FAVOR_ERR_UNSUPPORTED


@pytest.mark.parametrize("mode", ["bidir", "causal"])
def test_smreg_projections(mode):
    """Regularized rows (length sqrt(d), §2.3 SMREG) on the tensor-core shape."""
    shape = SHAPES[0]
    w, omega, q, k, v, f = _setup(shape, "softmax_pos", 1100, 57, regularized=True)
    np.testing.assert_allclose(np.linalg.norm(omega.astype(np.float64), axis=-1), np.sqrt(w.d), rtol=1e-2)
    with f:
        out = to_host(f.attn(*(to_dev(a, w.dtype) for a in (q, k, v)), causal=(mode == "causal")))
    ref = (O.favor_causal if mode == "causal" else O.favor_bidir)(q, k, v, omega, w.data_scale)
    assert O.row_rel_err(out, ref) <= TOL[w.dtype]
