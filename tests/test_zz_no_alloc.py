"""favor_attn_bidir_noalloc: the handle-free bidirectional call that runs on the
library's fixed device scratch array.  It must agree with favor_attn_bidir (the
handle path) within the dtype's tolerance on two calls in a row, and reject
sizes the fixed scratch cannot hold before launching anything.

The file name sorts last so that the GPU test also runs after every other
test has used the library on the same device."""
import numpy as np
import pytest

import oracle as O
import random_feature_gb300 as R
from random_feature_gb300 import build as _build
from synth import CONFIGS, make_workload

from _util import TOL, to_dev, to_host


@pytest.fixture(scope="module", autouse=True)
def _built_library():
    _build.build()


def test_rejects_sizes_beyond_fixed_scratch():
    # 64 heads x 256 features x 129 value columns x 2 state copies > 4,194,304 floats.
    # Checked on the host before any CUDA call, so this runs without a GPU.
    with pytest.raises(R.FavorError) as e:
        R.favor_attn_bidir_noalloc(1, 64, 256, 64, 128, "softmax_pos", "bf16", 0.35, 1, 1, 1, 1, 1, 128, stream=0)
    assert e.value.status == R.FAVOR_ERR_UNSUPPORTED
    assert "fixed scratch" in R.favor_last_error()


def test_rejects_null_omega():
    with pytest.raises(R.FavorError) as e:
        R.favor_attn_bidir_noalloc(0, 2, 64, 32, 32, "relu", "f32", 1.0, 1, 1, 1, 1, 1, 128, stream=0)
    assert e.value.status == R.FAVOR_ERR_INVALID_ARG


def test_rejects_misaligned_omega():
    """An omega address off a 16-byte boundary is refused before any launch
    (the kernels read omega rows as 16-byte vectors)."""
    n0 = R.favor_launch_count()
    with pytest.raises(R.FavorError) as e:
        R.favor_attn_bidir_noalloc(4, 2, 64, 32, 32, "softmax_pos", "f32", 1.0, 1, 1, 1, 1, 1, 128, stream=0)
    assert e.value.status == R.FAVOR_ERR_INVALID_ARG
    assert "aligned" in R.favor_last_error()
    assert R.favor_launch_count() == n0


def test_rejects_host_omega():
    """A host buffer (16-byte aligned) is not device memory: refused before any
    launch, on a machine with or without a GPU."""
    om = np.zeros(2 * 64 * 32 + 16, dtype=np.float32)
    addr = om.ctypes.data
    addr += (-addr) % 16
    n0 = R.favor_launch_count()
    with pytest.raises(R.FavorError) as e:
        R.favor_attn_bidir_noalloc(addr, 2, 64, 32, 32, "softmax_pos", "f32", 1.0, 1, 1, 1, 1, 1, 128, stream=0)
    assert e.value.status == R.FAVOR_ERR_INVALID_ARG
    assert "device" in R.favor_last_error()
    assert R.favor_launch_count() == n0


CASES = [
    # (config, overrides, kind): the tensor-core shape in bf16, with a split narrowed
    # to fit the scratch (B*H = 32, m = 256, dv = 64 leaves room for 6 segments per head),
    # and an fp32 shape on the CUDA-core path with a ragged tail.
    ("bidir_bf16", dict(B=2, H=16, L=4096), "softmax_pos"),
    ("bidir_bf16", dict(B=1, H=3, L=1000), "relu"),
    ("approx_f32", dict(B=2, H=4, L=777), "softmax_pos"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,over,kind", CASES)
def test_noalloc_matches_handle_path_twice(name, over, kind):
    import torch

    w = CONFIGS[name].replace(**over)
    omega, q, k, v = make_workload(w, 11)
    qd, kd, vd = (to_dev(a, w.dtype) for a in (q, k, v))
    with R.Favor(w.H, w.m, w.d, w.dv, kind, w.dtype, omega, w.data_scale, w.B, w.L) as f:
        ref = to_host(f.attn(qd, kd, vd, causal=False))
    # The handle path rounds omega to bf16 for the bf16 dtype; hand the same values over.
    om = omega.astype(np.float32)
    if w.dtype == "bf16":
        om = torch.from_numpy(om).to(torch.bfloat16).to(torch.float32).numpy()
    om_d = torch.from_numpy(np.ascontiguousarray(om)).cuda()
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    outs = []
    for _ in range(2):
        out = torch.full((w.B, w.H, w.L, w.dv), float("nan"), dtype=tdt, device="cuda")
        R.favor_attn_bidir_noalloc(om_d, w.H, w.m, w.d, w.dv, kind, w.dtype, w.data_scale, qd, kd, vd, out,
                                   w.B, w.L)
        torch.cuda.synchronize()
        outs.append(to_host(out))
    exact = O.favor_bidir(q, k, v, omega, w.data_scale, kind)
    for got in outs:
        assert np.isfinite(got).all()
        assert O.row_rel_err(got, ref) <= TOL[w.dtype]
        assert O.row_rel_err(got, exact) <= TOL[w.dtype]
    # Same inputs, same fixed work split: the two calls agree bit for bit.
    assert np.array_equal(outs[0], outs[1])
