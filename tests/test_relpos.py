"""GPU parity of the decaying causal state (RFA-Gate gates, PermuteFormer r)
and of PermuteFormer's position-dependent feature permutation, against the
float64 oracle; plus the argument checks of favor_set_relpos."""
import numpy as np
import pytest

import oracle as O
import random_feature_gb300 as R
from synth import CONFIGS, make_workload

from _util import TOL, to_dev, to_host
from test_variants import trig_row_condition

pytestmark = pytest.mark.gpu

SHAPES = [
    ("d64_m256_bf16", "bidir_bf16", dict(B=2, H=2)),
    ("d32_m48_bf16", "bidir_bf16", dict(B=1, H=3, d=32, dv=16, m=48)),
    ("d16_m64_f32", "approx_f32", dict(B=2, H=2, m=64, dv=32)),
]


def _setup(shape, kind, L, seed):
    _, base, over = shape
    w = CONFIGS[base].replace(L=L, **over)
    omega, q, k, v = make_workload(w, seed)
    f = R.Favor(w.H, w.m, w.d, w.dv, kind, w.dtype, omega, w.data_scale, w.B, w.L)
    return w, omega, q, k, v, f


def _gates(w, seed, lo=0.8, hi=1.0):
    return np.random.default_rng(seed).uniform(lo, hi, (w.B, w.H, w.L)).astype(np.float32)


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("kind", O.KINDS)
def test_gated_causal(shape, kind):
    # 1100 tokens: several segments, so the segment states are combined through gate products
    w, omega, q, k, v, f = _setup(shape, kind, 1100, 61)
    g = _gates(w, 61)
    import torch
    with f:
        out = to_host(f.attn_causal_gated(*(to_dev(a, w.dtype) for a in (q, k, v)),
                                          torch.from_numpy(g).cuda()))
    ref = O.favor_causal_gated(q, k, v, g, omega, w.data_scale, kind)
    assert O.row_rel_err(out, ref) <= TOL[w.dtype]


def test_gated_causal_fast_decay():
    """Gates near 0.3: the history fades within a few tokens and the segment
    products underflow to 0 without harm."""
    shape = SHAPES[0]
    w, omega, q, k, v, f = _setup(shape, "softmax_pos", 900, 62)
    g = _gates(w, 62, 0.1, 0.5)
    import torch
    with f:
        out = to_host(f.attn_causal_gated(*(to_dev(a, w.dtype) for a in (q, k, v)), torch.from_numpy(g).cuda()))
    ref = O.favor_causal_gated(q, k, v, g, omega, w.data_scale)
    assert np.isfinite(out).all()
    assert O.row_rel_err(out, ref) <= TOL[w.dtype]


@pytest.mark.parametrize("kind", O.KINDS)
@pytest.mark.parametrize("lo,hi", [(0.8, 1.0), (0.05, 0.6)], ids=["slow", "fast"])
def test_gated_causal_many_chunks_per_range(kind, lo, hi):
    """The tensor-core shape with several 128-token chunks per work range and a
    ragged tail (2 heads x 38491 tokens: 301 tiles a head, ranges of 4 tiles,
    so one range holds the end of head 0 and the start of head 1): the gated
    state is carried from chunk to chunk inside a range (decayed in place), from
    range to range (the decayed prefix of the pieces) and restarts at the head
    boundary inside a range.  Fast-decaying gates reach the 2^-126 clamp within
    a chunk."""
    import torch
    w = CONFIGS["bidir_bf16"].replace(B=1, H=2, L=38491)
    omega, q, k, v = make_workload(w, 64)
    g = _gates(w, 64, lo, hi)
    with R.Favor(w.H, w.m, w.d, w.dv, kind, w.dtype, omega, w.data_scale, w.B, w.L) as f:
        out = to_host(f.attn_causal_gated(*(to_dev(a, w.dtype) for a in (q, k, v)), torch.from_numpy(g).cuda()))
        assert R.favor_device_error(f.handle) == 0
    ref = O.favor_causal_gated(q, k, v, g, omega, w.data_scale, kind)
    assert np.isfinite(out).all()
    assert O.row_rel_err(out, ref) <= TOL[w.dtype]


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_gated_steps_continue_a_state(shape):
    """Gated decode steps in blocks of 1, 5 and 34 tokens from a zero state give
    the gated causal attention of the 40 tokens."""
    import torch
    w, omega, q, k, v, f = _setup(shape, "softmax_pos", 40, 63)
    g = _gates(w, 63, 0.5, 1.0)
    ref = O.favor_causal_gated(q, k, v, g, omega, w.data_scale)
    with f:
        st = f.new_state(w.B)
        outs = []
        t = 0
        for n in (1, 5, 34):
            sl = slice(t, t + n)
            outs.append(to_host(f.causal_step_gated(*(to_dev(a[:, :, sl], w.dtype) for a in (q, k, v)),
                                                    torch.from_numpy(np.ascontiguousarray(g[:, :, sl])).cuda(), st)))
            t += n
    assert O.row_rel_err(np.concatenate(outs, axis=2), ref) <= TOL[w.dtype]


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("kind", O.KINDS)
@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_permuteformer(shape, kind, causal):
    w, omega, q, k, v, f = _setup(shape, kind, 1100, 64)
    rng = np.random.default_rng(64)
    perm = np.stack([rng.permutation(w.m) for _ in range(w.H)]).astype(np.int32)
    r = rng.uniform(0.95, 0.999, w.H).astype(np.float32)
    with f:
        f.set_relpos(perm, r)
        out = to_host(f.attn(*(to_dev(a, w.dtype) for a in (q, k, v)), causal=causal))
    ref = O.favor_permute(q, k, v, omega, w.data_scale, perm, r, causal, kind)
    assert O.row_rel_err(out, ref) <= TOL[w.dtype]


def test_relpos_checks_and_clearing():
    import torch
    shape = SHAPES[0]
    w, omega, q, k, v, f = _setup(shape, "softmax_pos", 256, 65)
    with f:
        bad = np.tile(np.arange(w.m, dtype=np.int32), (w.H, 1))
        bad[1, 3] = 4                       # duplicate: not a permutation
        with pytest.raises(R.FavorError) as ei:
            f.set_relpos(bad, None)
        assert ei.value.status == R.FAVOR_ERR_INVALID_ARG
        with pytest.raises(R.FavorError) as ei:
            f.set_relpos(None, np.array([0.5, 1.5], np.float32))
        assert ei.value.status == R.FAVOR_ERR_INVALID_ARG
        dev = [to_dev(a, w.dtype) for a in (q, k, v)]
        plain = to_host(f.attn(*dev, causal=True))
        perm = np.stack([np.random.default_rng(h).permutation(w.m) for h in range(w.H)]).astype(np.int32)
        f.set_relpos(perm, None)
        for call in (lambda: f.kv_state(dev[1], dev[2]),
                     lambda: f.attn_backward(*dev, dev[2]),
                     lambda: f.attn_causal_gated(*dev, torch.ones((w.B, w.H, w.L), device="cuda"))):
            with pytest.raises(R.FavorError) as ei:
                call()
            assert ei.value.status == R.FAVOR_ERR_UNSUPPORTED
        f.set_relpos(None, None)            # cleared: the plain (tensor-core) path again
        again = to_host(f.attn(*dev, causal=True))
        np.testing.assert_array_equal(again, plain)


def test_variants_full_size_sampled_heads():
    """The bench workload (B=1, H=16, L=65536, bf16) through the calls the
    bench's variants line times; the oracle recomputes heads 0 and 9."""
    import torch
    w = CONFIGS["long_bf16"]
    omega, q, k, v = make_workload(w, 0)
    heads = [0, 9]
    sel = lambda a: np.ascontiguousarray(a[:, heads])
    dev = [to_dev(a, w.dtype) for a in (q, k, v)]
    rng = np.random.default_rng(3)
    gate = rng.uniform(0.8, 1.0, (w.B, w.H, w.L)).astype(np.float32)
    perm = np.stack([rng.permutation(w.m) for _ in range(w.H)]).astype(np.int32)
    r = np.full(w.H, 0.999, np.float32)
    half = np.ascontiguousarray(omega[:, : w.m // 2])
    cases = [
        ("softmax_hyp", half, "causal", lambda: O.favor_causal(sel(q), sel(k), sel(v), half[heads], w.data_scale,
                                                               "softmax_hyp")),
        ("softmax_trig", half, "causal", lambda: O.favor_causal(sel(q), sel(k), sel(v), half[heads], w.data_scale,
                                                                "softmax_trig")),
        ("softmax_pos", omega, "gate", lambda: O.favor_causal_gated(sel(q), sel(k), sel(v), sel(gate), omega[heads],
                                                                    w.data_scale)),
        ("softmax_pos", omega, "relpos", lambda: O.favor_permute(sel(q), sel(k), sel(v), omega[heads], w.data_scale,
                                                                 perm[heads], r[heads], True)),
    ]
    for kind, om, mode, ref_fn in cases:
        with R.Favor(w.H, w.m, w.d, w.dv, kind, w.dtype, om, w.data_scale, w.B, w.L) as f:
            if mode == "gate":
                out = f.attn_causal_gated(*dev, torch.from_numpy(gate).cuda())
            else:
                if mode == "relpos":
                    f.set_relpos(perm, r)
                out = f.attn(*dev, causal=True)
            got = to_host(out[:, heads])
        ref = ref_fn()
        assert O.row_rel_err(got, ref) <= TOL[w.dtype], (kind, mode)


@pytest.mark.parametrize("L", [1, 127, 129, 300])
def test_tensor_core_variants_short_and_ragged(L):
    """Trigonometric (bidirectional and causal) and gated calls on the tensor-core
    shape at one token, one chunk short of full, one token past a chunk and a
    ragged multi-chunk length: rows past L must neither leak into the sums nor
    be written, for the sin/cos epilogue, the key factors h(s k) and the gates'
    scan alike."""
    import torch
    w = CONFIGS["bidir_bf16"].replace(B=2, H=3, L=L)
    omega, q, k, v = make_workload(w, 65)
    half = np.ascontiguousarray(omega[:, : w.m // 2])
    dev = [to_dev(a, w.dtype) for a in (q, k, v)]
    with R.Favor(w.H, w.m, w.d, w.dv, "softmax_trig", w.dtype, half, w.data_scale, w.B, w.L) as f:
        for causal in (False, True):
            out = to_host(f.attn(*dev, causal=causal))
            ref = (O.favor_causal if causal else O.favor_bidir)(q, k, v, half, w.data_scale, "softmax_trig")
            assert np.isfinite(out).all()
            scale = np.maximum(np.abs(ref).max(axis=-1), 1e-300)
            err = np.abs(out - ref).max(axis=-1) / scale
            # bf16 operands amplified by each row's cancellation (as test_variants.assert_trig_rows)
            cond = trig_row_condition(q, k, v, half, w.data_scale, causal)
            assert np.all(err <= TOL[w.dtype] + 4 * 2.0 ** -9 * cond), (causal, float(np.max(err)))
        assert R.favor_device_error(f.handle) == 0
    g = _gates(w, 65, 0.3, 1.0)
    for kind in O.KINDS:
        with R.Favor(w.H, w.m, w.d, w.dv, kind, w.dtype, omega, w.data_scale, w.B, w.L) as f:
            out = to_host(f.attn_causal_gated(*dev, torch.from_numpy(g).cuda()))
            assert R.favor_device_error(f.handle) == 0
        ref = O.favor_causal_gated(q, k, v, g, omega, w.data_scale, kind)
        assert np.isfinite(out).all()
        assert O.row_rel_err(out, ref) <= TOL[w.dtype], (kind, L)
