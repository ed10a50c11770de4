"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/favor.h declares, and rejects bad arguments before
touching a device."""
import ctypes
import os
import re

import numpy as np
import pytest

import random_feature_gb300 as R
from random_feature_gb300 import build as _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built_library():
    _build.build()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "favor.h")).read()
    return set(re.findall(r"FAVOR_API\s+[\w\s\*]+?\b(favor_\w+)\s*\(", text))


def test_library_builds_and_exports_header_symbols():
    declared = _declared_symbols()
    assert {"favor_create", "favor_feature_map", "favor_attn_bidir", "favor_attn_causal",
            "favor_destroy"} <= declared
    L = R.lib()
    for name in declared:
        assert hasattr(L, name), name
    assert declared == set(R.EXPORTED_SYMBOLS)


def test_status_strings():
    assert R.favor_status_str(R.FAVOR_OK) == "FAVOR_OK"
    assert R.favor_status_str(R.FAVOR_ERR_UNSUPPORTED) == "FAVOR_ERR_UNSUPPORTED"
    assert R.favor_status_str(99) == "FAVOR_ERR_UNKNOWN"


def _raw_create(H=1, m=32, d=16, dv=16, kind=0, dtype=0, omega=True, s=1.0, max_B=1, max_L=64, out=True):
    L = R.lib()
    h = ctypes.c_void_p(12345)
    om = np.zeros((H, m, d), np.float32) if omega else None
    ptr = om.ctypes.data_as(ctypes.POINTER(ctypes.c_float)) if omega else None
    st = L.favor_create(ctypes.byref(h) if out else None, H, m, d, dv, kind, dtype, ptr, s, max_B, max_L)
    return st, h.value


@pytest.mark.parametrize("kw,want", [
    (dict(out=False), R.FAVOR_ERR_INVALID_ARG),
    (dict(omega=False), R.FAVOR_ERR_INVALID_ARG),
    (dict(H=0), R.FAVOR_ERR_INVALID_ARG),
    (dict(max_L=0), R.FAVOR_ERR_INVALID_ARG),
    (dict(kind=7), R.FAVOR_ERR_INVALID_ARG),
    (dict(dtype=5), R.FAVOR_ERR_INVALID_ARG),
    (dict(s=0.0), R.FAVOR_ERR_INVALID_ARG),
    (dict(s=float("nan")), R.FAVOR_ERR_INVALID_ARG),
    (dict(d=48), R.FAVOR_ERR_UNSUPPORTED),
    (dict(dv=8), R.FAVOR_ERR_UNSUPPORTED),
    (dict(m=24), R.FAVOR_ERR_UNSUPPORTED),
    (dict(m=512), R.FAVOR_ERR_UNSUPPORTED),
    (dict(m=0), R.FAVOR_ERR_INVALID_ARG),
    (dict(d=0), R.FAVOR_ERR_INVALID_ARG),
    (dict(dv=0), R.FAVOR_ERR_INVALID_ARG),
    (dict(max_B=0), R.FAVOR_ERR_INVALID_ARG),
    # max_B * H * max_L * max(d, dv) above 2^40: refused before any allocation
    (dict(max_B=1 << 20, max_L=1 << 20), R.FAVOR_ERR_UNSUPPORTED),
])
def test_create_rejects_bad_arguments(kw, want):
    st, h = _raw_create(**kw)
    assert st == want, R.favor_last_error()
    assert R.favor_last_error()
    if kw.get("out", True):
        assert h is None          # *out is cleared on failure


def test_calls_reject_null_handle():
    L = R.lib()
    assert L.favor_attn_bidir(None, 1, 1, 1, 1, 1, 1, None) == R.FAVOR_ERR_INVALID_ARG
    assert L.favor_attn_causal(None, 1, 1, 1, 1, 1, 1, None) == R.FAVOR_ERR_INVALID_ARG
    assert L.favor_feature_map(None, 1, 1, 1, 1, None) == R.FAVOR_ERR_INVALID_ARG
    assert L.favor_destroy(None) == R.FAVOR_OK


def test_stateful_backward_variant_calls_reject_null_handle():
    """Every call past the forward ones checks its handle first (no CUDA call)."""
    L = R.lib()
    bad = R.FAVOR_ERR_INVALID_ARG
    assert L.favor_kv_state(None, 1, 1, 1, 1, 1, None) == bad
    assert L.favor_attn_from_state(None, 1, 1, 1, 1, 1, None) == bad
    assert L.favor_attn_causal_step(None, 1, 1, 1, 1, 1, 1, 1, None) == bad
    assert L.favor_attn_bidir_backward(None, 1, 1, 1, 1, 1, 1, 1, 1, 1, None) == bad
    assert L.favor_attn_causal_backward(None, 1, 1, 1, 1, 1, 1, 1, 1, 1, None) == bad
    assert L.favor_attn_causal_gated(None, 1, 1, 1, 1, 1, 1, 1, None) == bad
    assert L.favor_attn_causal_step_gated(None, 1, 1, 1, 1, 1, 1, 1, 1, None) == bad
    assert L.favor_set_relpos(None, None, None) == bad


def test_launch_counter_is_monotone():
    a = R.favor_launch_count()
    assert R.favor_launch_count() >= a >= 0


def test_python_binding_has_c_names():
    for name in R.EXPORTED_SYMBOLS:
        assert callable(getattr(R, name))


def test_bench_algorithmic_counts():
    """The bench's per-token*head work counts, against hand arithmetic for the
    bench shape (d = dv = 64, m = 256, bf16)."""
    import bench
    from synth import CONFIGS
    w = CONFIGS["long_bf16"]
    b, f, e = bench.per_token_head(w, "causal_chunks", "softmax_pos")
    assert (b, f, e) == ((2 * 64 + 2 * 64) * 2, 4 * 256 * 64 + 4 * 256 * 65, 2 * 256)
    b, f, e = bench.per_token_head(w, "bidir_readout", "relu")
    assert (b, f, e) == ((64 + 64) * 2, 2 * 256 * 64 + 2 * 256 * 65, 0)
    assert bench.backward_flops_per_token_head(w) == 8 * 256 * 64 + 6 * 256 * 65 + 4 * 256 * 64 == 296448


def test_bench_cpu_model_names_the_host():
    """The oracle baseline names the host CPU (model name, or the Arm
    implementer/part codes when /proc/cpuinfo has no model name)."""
    import bench
    name = bench.cpu_model()
    assert isinstance(name, str) and name.strip() and name != "unknown"


def test_bench_reference_arm_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the contract's keys; tiny workload, one step."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_f32", "--steps", "1", "--warmup", "0"], capture_output=True, text=True, cwd=root,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
