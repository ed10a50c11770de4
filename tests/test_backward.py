"""GPU parity of the backward calls (dq, dk, dv of the bidirectional and causal
attention) against the float64 oracle's exact derivative.

Error measure for a gradient tensor: per (b, h) slice, max over rows i of
max_c |g_ic - o_ic| / max(max_c |o_ic|, 1e-3 * max |o| over the slice).  The
slice floor covers rows whose gradient vanishes by structure (causal query 0:
out_0 = v_0 whatever q_0, so dq_0 = 0 exactly and the device returns rounding
noise there).

Tolerances: bf16 2e-2 as for the forward.  fp32 1e-3, ten times the forward's:
the step dphi_r = (u_r - z_r (dO . out)) / den subtracts two nearly equal
terms (their difference is sum_j phi_j[r] (v_j - out) . dO); over the shapes
below its condition number reaches 3.2e3 (d = 128, positive features), so
fp32 rounding alone gives up to 2^-24 * 3.2e3 = 1.9e-4, and 1e-3 leaves a 5x
margin.  Every other step of dq, dk, dv has condition below 10.
"""
import numpy as np
import pytest

import oracle as O
import random_feature_gb300 as R
from synth import CONFIGS, make_upstream_grad, make_workload

from _util import to_dev, to_dev_unaligned, to_host

TOL_GRAD = {"f32": 1e-3, "bf16": 2e-2}

SHAPES = [
    # (name, base config, overrides): the tensor-core forward shape, CUDA-core
    # shapes with m not a multiple of 32, dv = 128 (16-token tiles), fp32
    ("d64_m256_bf16", "bidir_bf16", dict(B=2, H=2)),
    ("d32_m48_bf16", "bidir_bf16", dict(B=1, H=3, d=32, dv=16, m=48)),
    ("d16_m64_f32", "approx_f32", dict(B=2, H=2, m=64, dv=32)),
    ("d128_dv128_f32", "approx_f32", dict(B=1, H=2, d=128, dv=128, m=256)),
]


def grad_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    B, H = ref.shape[:2]
    worst = 0.0
    for b in range(B):
        for h in range(H):
            g, o = got[b, h], ref[b, h]
            floor = 1e-3 * np.max(np.abs(o))
            scale = np.maximum(np.max(np.abs(o), axis=1), floor)
            scale = np.where(scale > 0, scale, 1.0)
            worst = max(worst, float(np.max(np.abs(g - o).max(axis=1) / scale)))
    return worst


def relu_kink_rows_ok(got, ref, x, omega, dphi, s, tol):
    """Rows of a ReLU gradient dx (one head) checked with the kink allowed both ways.

    The derivative of max(u, 0) at u = 0 is a choice, and a projection
    omega_r . x within fp32 rounding of 0 can fall on either side on the
    device and in the float64 oracle.  For rows that hold such features
    (|omega_r . x| below 4 * 64 * 2^-24 * sum_c |omega_rc x_c|), every
    combination of their mask bits is a valid gradient: the row passes if the
    device matches any of them.  Other rows must match the oracle as usual.
    Returns the number of rows that match no valid gradient."""
    m = omega.shape[0]
    proj = x @ omega.T
    band = 4 * 64 * 2.0 ** -24 * (np.abs(x) @ np.abs(omega).T)
    amb = np.abs(proj) < band
    floor = 1e-3 * np.max(np.abs(ref))
    bad = 0
    for i in range(ref.shape[0]):
        scale = max(np.max(np.abs(ref[i])), floor) or 1.0
        if np.max(np.abs(got[i] - ref[i])) / scale <= tol:
            continue
        rs = np.nonzero(amb[i])[0]
        if len(rs) == 0 or len(rs) > 4:
            bad += 1
            continue
        ok = False
        for bits in range(1, 1 << len(rs)):
            alt = ref[i].copy()
            for t, r in enumerate(rs):
                if bits >> t & 1:   # flip feature r's mask relative to the oracle's decision
                    sign = -1.0 if proj[i, r] > 0 else 1.0
                    alt += sign * s * dphi[i, r] * omega[r] / np.sqrt(m)
            if np.max(np.abs(got[i] - alt)) / scale <= tol:
                ok = True
                break
        bad += 0 if ok else 1
    return bad


def check_grads(w, kind, causal, got, ref, q, k, v, g, omega):
    """dq, dk, dv against the oracle.  ReLU dq and dk go row by row, with
    projections on the kink allowed either way; dv has no kink dependence
    (phi_k is continuous there)."""
    assert grad_err(got[2], ref[2]) <= TOL_GRAD[w.dtype], "dv"
    if kind != "relu":
        for name, a, b in zip(("dq", "dk"), got[:2], ref[:2]):
            assert grad_err(a, b) <= TOL_GRAD[w.dtype], name
        return
    vjp = O.attn_from_features_causal_vjp if causal else O.attn_from_features_bidir_vjp
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            x = w.data_scale * q[b, h].astype(np.float64)
            y = w.data_scale * k[b, h].astype(np.float64)
            om = omega[h].astype(np.float64)
            pq, pk = O.feature_map(x, om, kind), O.feature_map(y, om, kind)
            dpq, dpk, _ = vjp(pq, pk, v[b, h], g[b, h])
            tol = TOL_GRAD[w.dtype]
            assert relu_kink_rows_ok(got[0][b, h], ref[0][b, h], x, om, dpq, w.data_scale, tol) == 0, ("dq", b, h)
            assert relu_kink_rows_ok(got[1][b, h], ref[1][b, h], y, om, dpk, w.data_scale, tol) == 0, ("dk", b, h)


def _run(shape, kind, causal, L, seed):
    _, base, over = shape
    w = CONFIGS[base].replace(L=L, **over)
    omega, q, k, v = make_workload(w, seed)
    g = make_upstream_grad(w, seed)
    bwd = O.favor_causal_backward if causal else O.favor_bidir_backward
    ref = bwd(q, k, v, g, omega, w.data_scale, kind)
    with R.Favor(w.H, w.m, w.d, w.dv, kind, w.dtype, omega, w.data_scale, w.B, w.L) as f:
        dev = [to_dev(a, w.dtype) for a in (q, k, v, g)]
        got = f.attn_backward(*dev, causal=causal)
        got = [to_host(t) for t in got]
        assert R.favor_device_error(f.handle) == 0
    return w, got, ref


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("kind", O.KINDS)
@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_backward_matches_oracle(shape, kind, causal):
    # 1100 tokens: several 128-token segments per head and a ragged last tile
    L = 1100 if shape[0] != "d128_dv128_f32" else 333
    w, got, ref = _run(shape, kind, causal, L, 31)
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        e = grad_err(a, b)
        assert e <= TOL_GRAD[w.dtype], (name, e)


@pytest.mark.gpu
@pytest.mark.parametrize("L", [2, 31, 33])
def test_backward_short_sequences(L):
    shape = SHAPES[0]
    for causal in (False, True):
        w, got, ref = _run(shape, "softmax_pos", causal, L, 32 + L)
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert grad_err(a, b) <= TOL_GRAD[w.dtype], (name, causal, L)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_backward_single_token_is_identity_on_v(causal):
    """L = 1: out = v whatever q and k, so dv = dO and dq = dk = 0 (the device
    returns rounding noise for the zero gradients)."""
    w, got, ref = _run(SHAPES[2], "softmax_pos", causal, 1, 40)
    np.testing.assert_allclose(got[2], ref[2], rtol=1e-6, atol=1e-6)
    assert np.max(np.abs(got[0])) < 1e-5 and np.max(np.abs(got[1])) < 1e-5


@pytest.mark.gpu
def test_backward_is_deterministic():
    shape = SHAPES[0]
    _, base, over = shape
    w = CONFIGS[base].replace(L=900, **over)
    omega, q, k, v = make_workload(w, 41)
    g = make_upstream_grad(w, 41)
    with R.Favor(w.H, w.m, w.d, w.dv, "softmax_pos", w.dtype, omega, w.data_scale, w.B, w.L) as f:
        dev = [to_dev(a, w.dtype) for a in (q, k, v, g)]
        a = [t.clone() for t in f.attn_backward(*dev, causal=True)]
        b = f.attn_backward(*dev, causal=True)
        for x, y in zip(a, b):
            assert bool((x == y).all())


@pytest.mark.gpu
def test_backward_argument_checks():
    shape = SHAPES[0]
    _, base, over = shape
    w = CONFIGS[base].replace(L=64, **over)
    omega, q, k, v = make_workload(w, 42)
    with R.Favor(w.H, w.m, w.d, w.dv, "softmax_pos", w.dtype, omega, w.data_scale, w.B, w.L) as f:
        dev = [to_dev(a, w.dtype) for a in (q, k, v, v)]
        dq, dk, dv = (to_dev(np.zeros_like(a), w.dtype) for a in (q, k, v))
        n0 = R.favor_launch_count()
        with pytest.raises(R.FavorError) as ei:
            R.favor_attn_bidir_backward(f.handle, *dev[:3], 0, dq, dk, dv, w.B, w.L)
        assert ei.value.status == R.FAVOR_ERR_INVALID_ARG
        with pytest.raises(R.FavorError) as ei:
            R.favor_attn_causal_backward(f.handle, *dev, dq, dk, dv, w.B, w.L + 1)
        assert ei.value.status == R.FAVOR_ERR_INVALID_ARG
        assert R.favor_launch_count() == n0


@pytest.mark.gpu
@pytest.mark.parametrize("kind", O.KINDS)
@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_backward_full_size_sampled_heads(causal, kind):
    """The bench workload (B=1, H=16, L=65536, bf16, d=dv=64, m=256) in the
    bench's launch configuration; the oracle recomputes heads 0 and 9."""
    import torch
    w = CONFIGS["long_bf16"]
    omega, q, k, v = make_workload(w, 0)
    g = make_upstream_grad(w, 0)
    with R.Favor(w.H, w.m, w.d, w.dv, kind, w.dtype, omega, w.data_scale, w.B, w.L) as f:
        dev = [to_dev(a, w.dtype) for a in (q, k, v, g)]
        got = f.attn_backward(*dev, causal=causal)
        torch.cuda.synchronize()
        assert R.favor_device_error(f.handle) == 0
        heads = [0, 9]
        got = [to_host(t[:, heads]) for t in got]
    sel = lambda a: np.ascontiguousarray(a[:, heads])
    ref = (O.favor_causal_backward if causal else O.favor_bidir_backward)(
        sel(q), sel(k), sel(v), sel(g), omega[heads], w.data_scale, kind)
    check_grads(w, kind, causal, got, ref, sel(q), sel(k), sel(v), sel(g), omega[heads])


@pytest.mark.gpu
@pytest.mark.parametrize("kind", O.KINDS)
@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_backward_ranges_cross_heads_with_ragged_tiles(kind, causal):
    """B=4, H=16, L=1100 on the tensor-core shape: 576 tiles over the SMs, so a
    CTA's range of tiles crosses head boundaries and every head ends in a
    ragged tile (the per-head operands reload mid-range, pieces are combined
    across CTAs; causal: the running prefix and suffix states are carried over
    several chunks inside a range and restart at each head)."""
    shape = ("d64_m256_bf16", "bidir_bf16", dict(B=4, H=16))
    w, got, ref = _run(shape, kind, causal, 1100, 77)
    omega, q, k, v = make_workload(w, 77)
    check_grads(w, kind, causal, got, ref, q, k, v, make_upstream_grad(w, 77), omega)


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["softmax_pos", "relu"])
def test_causal_backward_long_ranges(kind):
    """One head pair over 40 chunks (B=1, H=2, L=5000): every CTA range is a
    single chunk here, and with the sequence split over fewer CTAs (B=1, H=1,
    L=40000: 313 chunks, three per range) the states cross ranges both
    ways; both against the oracle."""
    for H, L in ((2, 5000), (1, 40000)):
        shape = ("d64_m256_bf16", "bidir_bf16", dict(B=1, H=H))
        w, got, ref = _run(shape, kind, True, L, 91 + H)
        omega, q, k, v = make_workload(w, 91 + H)
        check_grads(w, kind, True, got, ref, q, k, v, make_upstream_grad(w, 91 + H), omega)


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [SHAPES[0], SHAPES[2]], ids=[SHAPES[0][0], SHAPES[2][0]])
@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_backward_unaligned_inputs(shape, causal):
    """q, k, v, dO one element past a 16-byte boundary: tiles are staged with
    plain loads instead of asynchronous copies (and the tensor-core shape runs
    on the CUDA cores); same gradients."""
    _, base, over = shape
    w = CONFIGS[base].replace(L=700, **over)
    omega, q, k, v = make_workload(w, 23)
    g = make_upstream_grad(w, 23)
    bwd = O.favor_causal_backward if causal else O.favor_bidir_backward
    ref = bwd(q, k, v, g, omega, w.data_scale, "softmax_pos")
    with R.Favor(w.H, w.m, w.d, w.dv, "softmax_pos", w.dtype, omega, w.data_scale, w.B, w.L) as f:
        dev = [to_dev_unaligned(a, w.dtype) for a in (q, k, v, g)]
        got = [to_host(t) for t in f.attn_backward(*dev, causal=causal)]
        assert R.favor_device_error(f.handle) == 0
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        assert grad_err(a, b) <= TOL_GRAD[w.dtype], name


@pytest.mark.gpu
@pytest.mark.parametrize("kind,base,over", [
    ("softmax_pos", "causal_bf16", dict(B=1, H=2, L=1100)),
    ("relu", "causal_bf16", dict(B=1, H=2, L=1100)),
    ("softmax_pos", "bidir_bf16", dict(B=1, H=2, L=700, std=1.0)),
    ("relu", "bidir_bf16", dict(B=1, H=2, L=700, std=1.0)),
], ids=["sharp_keys-softmax_pos", "sharp_keys-relu", "wide_inputs-softmax_pos", "wide_inputs-relu"])
def test_causal_backward_feature_range(kind, base, over):
    """Inputs whose features span a wider range than the default workloads:
    the causal config's sharp key rows (1% of keys x4) and inputs at twice the
    default spread (sharper attention, so dq and dk cancel more).  The
    tensor-core causal backward takes the key features of its in-chunk
    products as bf16 pairs in the query pass and rounds the key pass's
    in-chunk term to f16 under power-of-two scales; the gradients must meet
    the bf16 bound against the oracle."""
    w = CONFIGS[base].replace(**over)
    omega, q, k, v = make_workload(w, 57)
    g = make_upstream_grad(w, 57)
    ref = O.favor_causal_backward(q, k, v, g, omega, w.data_scale, kind)
    with R.Favor(w.H, w.m, w.d, w.dv, kind, w.dtype, omega, w.data_scale, w.B, w.L) as f:
        dev = [to_dev(a, w.dtype) for a in (q, k, v, g)]
        got = [to_host(t) for t in f.attn_backward(*dev, causal=True)]
        assert R.favor_device_error(f.handle) == 0
    check_grads(w, kind, True, got, ref, q, k, v, g, omega)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_relu_backward_zero_denominator_rows(causal):
    """ReLU features of an all-zero query row are all zero, so its denominator
    is 0 and its output is 0 whatever v (the zero-denominator rule of the
    forward): its dq is 0, and it adds nothing to dk or dv.  Rows in the
    first chunk, in the middle and at the end of the sequence."""
    shape = SHAPES[0]
    _, base, over = shape
    w = CONFIGS[base].replace(L=700, **over)
    omega, q, k, v = make_workload(w, 61)
    g = make_upstream_grad(w, 61)
    zero_rows = [0, 5, 300, 699]
    q[:, :, zero_rows, :] = 0.0
    bwd = O.favor_causal_backward if causal else O.favor_bidir_backward
    ref = bwd(q, k, v, g, omega, w.data_scale, "relu")
    with R.Favor(w.H, w.m, w.d, w.dv, "relu", w.dtype, omega, w.data_scale, w.B, w.L) as f:
        dev = [to_dev(a, w.dtype) for a in (q, k, v, g)]
        got = [to_host(t) for t in f.attn_backward(*dev, causal=causal)]
        assert R.favor_device_error(f.handle) == 0
    assert np.all(got[0][:, :, zero_rows, :] == 0.0)
    check_grads(w, "relu", causal, got, ref, q, k, v, g, omega)
