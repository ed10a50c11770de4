"""Failure detection without a GPU fault: the kernels' waits are bounded, and a
wait that runs out writes a code to the handle's device error word, returns,
and leaves the context usable.  favor_check_bounded_wait runs one such wait
on an mbarrier phase that nothing completes (no copies, no tensor memory),
with a limit of a few thousand cycles."""
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


def test_check_refuses_null_handle_and_bad_limits():
    with pytest.raises(R.FavorError) as e:
        R.favor_check_bounded_wait(0, 5000, stream=0)
    assert e.value.status == R.FAVOR_ERR_INVALID_ARG


@pytest.mark.gpu
def test_bounded_wait_gives_up_and_reports():
    import torch

    w = CONFIGS["bidir_bf16"].replace(B=1, H=2, L=300)
    omega, q, k, v = make_workload(w, 4)
    with R.Favor(w.H, w.m, w.d, w.dv, "softmax_pos", w.dtype, omega, w.data_scale, w.B, w.L) as f:
        assert R.favor_device_error(f.handle) == 0
        for bad in (999, (1 << 24) + 1):
            with pytest.raises(R.FavorError) as e:
                R.favor_check_bounded_wait(f.handle, bad)
            assert e.value.status == R.FAVOR_ERR_INVALID_ARG
        n0 = R.favor_launch_count()
        R.favor_check_bounded_wait(f.handle, 20000)
        torch.cuda.synchronize()
        assert R.favor_launch_count() == n0 + 1
        assert R.favor_device_error(f.handle) == R.FAVOR_WAIT_CHECK_CODE
        # a second expiry keeps the first code
        R.favor_check_bounded_wait(f.handle, 5000)
        assert R.favor_device_error(f.handle) == R.FAVOR_WAIT_CHECK_CODE
    # the context is still usable: a fresh handle computes attention and reports no error
    with R.Favor(w.H, w.m, w.d, w.dv, "softmax_pos", w.dtype, omega, w.data_scale, w.B, w.L) as f:
        qd, kd, vd = (to_dev(a, w.dtype) for a in (q, k, v))
        got = to_host(f.attn(qd, kd, vd, causal=True))
        torch.cuda.synchronize()
        assert R.favor_device_error(f.handle) == 0
    assert O.row_rel_err(got, O.favor_causal(q, k, v, omega, w.data_scale)) <= TOL[w.dtype]
