"""GPU parity of the stateful calls (key/value state, readout from a state,
causal continuation from a state) against the float64 oracle, on the
tensor-core shape and on CUDA-core shapes, both feature kinds."""
import numpy as np
import pytest

import oracle as O
import random_feature_gb300 as R
from synth import CONFIGS, make_workload

from _util import TOL, to_dev, to_host

SHAPES = [
    # (name, base config, overrides)
    ("tc_bf16", "bidir_bf16", dict(B=2, H=3)),
    ("simt_bf16", "bidir_bf16", dict(B=1, H=2, d=32, dv=32, m=128)),
    ("simt_f32", "approx_f32", dict(B=2, H=2, m=64)),
]


def _setup(shape, kind, L, seed):
    _, base, over = shape
    w = CONFIGS[base].replace(L=L, **over)
    omega, q, k, v = make_workload(w, seed)
    f = R.Favor(w.H, w.m, w.d, w.dv, kind, w.dtype, omega, w.data_scale, w.B, w.L)
    return w, omega, q, k, v, f


def _kappa(omega):
    sq = np.max(np.sum(np.asarray(omega, np.float64) ** 2, axis=-1), axis=-1)   # [H]
    return np.maximum(0.0, 0.5 * sq - 60.0)


def _state_err(got, ref):
    # row-normwise over the (S_r, z_r) rows of every head
    return O.row_rel_err(got.reshape(-1, got.shape[-1]), ref.reshape(-1, ref.shape[-1]))


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("kind", O.KINDS)
def test_kv_state_and_chunked_accumulation(shape, kind):
    w, omega, q, k, v, f = _setup(shape, kind, 1000, 21)
    with f:
        kd, vd = to_dev(k, w.dtype), to_dev(v, w.dtype)
        st = to_host(f.kv_state(kd, vd))
        ref = O.favor_kv_state(k, v, omega, w.data_scale, kind) * np.exp(-_kappa(omega))[None, :, None, None]
        assert _state_err(st, ref) <= TOL[w.dtype]
        # two chunks accumulate into the same state
        s2 = f.kv_state(to_dev(k[:, :, :377], w.dtype), to_dev(v[:, :, :377], w.dtype))
        f.kv_state(to_dev(k[:, :, 377:], w.dtype), to_dev(v[:, :, 377:], w.dtype), state=s2)
        assert _state_err(to_host(s2), ref) <= TOL[w.dtype]


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("kind", O.KINDS)
def test_cross_attention_from_state(shape, kind):
    # keys / values of one sequence (700 tokens), queries of another (300 tokens)
    w, omega, q, k, v, f = _setup(shape, kind, 700, 22)
    _, q2, _, _ = make_workload(w.replace(L=300), 23)
    with f:
        st = f.kv_state(to_dev(k, w.dtype), to_dev(v, w.dtype))
        got = to_host(f.attn_from_state(to_dev(q2, w.dtype), st))
        ref = O.favor_attn_from_state(q2, O.favor_kv_state(k, v, omega, w.data_scale, kind), omega, w.data_scale, kind)
        assert O.row_rel_err(got, ref) <= TOL[w.dtype]


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("kind", O.KINDS)
def test_causal_steps_chain_to_full_causal(shape, kind):
    w, omega, q, k, v, f = _setup(shape, kind, 300, 24)
    with f:
        qd, kd, vd = (to_dev(a, w.dtype) for a in (q, k, v))
        state = f.new_state(w.B)
        outs, t0 = [], 0
        for T in (1, 5, 130, 64, 100):
            outs.append(to_host(f.causal_step(qd[:, :, t0:t0 + T].contiguous(), kd[:, :, t0:t0 + T].contiguous(),
                                              vd[:, :, t0:t0 + T].contiguous(), state)))
            t0 += T
        got = np.concatenate(outs, axis=2)
        ref = O.favor_causal(q, k, v, omega, w.data_scale, kind)
        assert O.row_rel_err(got, ref) <= TOL[w.dtype]
        assert O.row_rel_err(got, to_host(f.attn(qd, kd, vd, causal=True))) <= 2 * TOL[w.dtype]
        ref_state = O.favor_kv_state(k, v, omega, w.data_scale, kind) * np.exp(-_kappa(omega))[None, :, None, None]
        assert _state_err(to_host(state), ref_state) <= TOL[w.dtype]


@pytest.mark.gpu
@pytest.mark.parametrize("kind", O.KINDS)
def test_decode_tokens_after_prefill_state(kind):
    # prefill 900 tokens into a state with the tensor-core path, then decode 12 tokens one at a time
    shape = SHAPES[0]
    w, omega, q, k, v, f = _setup(shape, kind, 912, 25)
    with f:
        state = f.kv_state(to_dev(k[:, :, :900], w.dtype), to_dev(v[:, :, :900], w.dtype))
        outs = []
        for t in range(900, 912):
            outs.append(to_host(f.causal_step(to_dev(q[:, :, t:t + 1], w.dtype), to_dev(k[:, :, t:t + 1], w.dtype),
                                              to_dev(v[:, :, t:t + 1], w.dtype), state)))
        got = np.concatenate(outs, axis=2)
        ref = O.favor_causal(q, k, v, omega, w.data_scale, kind)[:, :, 900:]
        assert O.row_rel_err(got, ref) <= TOL[w.dtype]
