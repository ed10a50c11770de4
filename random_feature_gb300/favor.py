"""ctypes binding of the FAVOR+ C ABI (include/favor.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libfavor.so.  The functions keep the C names; tensors may be torch
CUDA tensors (their data_ptr() is passed) or raw integer device addresses.
The stream defaults to torch's current stream on the tensor's device.

If the shared library has not been built, importing works but the first call
raises ``FavorLibraryMissing`` -- there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "FAVOR_OK", "FAVOR_ERR_INVALID_ARG", "FAVOR_ERR_UNSUPPORTED", "FAVOR_ERR_NOMEM", "FAVOR_ERR_CUDA",
    "FAVOR_KERNEL_SOFTMAX_POS", "FAVOR_KERNEL_RELU", "FAVOR_KERNEL_SOFTMAX_HYP", "FAVOR_KERNEL_SOFTMAX_TRIG",
    "FAVOR_DTYPE_F32", "FAVOR_DTYPE_BF16",
    "FavorError", "FavorLibraryMissing", "lib", "lib_path",
    "favor_create", "favor_feature_map", "favor_attn_bidir", "favor_attn_causal", "favor_destroy",
    "favor_status_str", "favor_last_error", "favor_launch_count", "Favor", "EXPORTED_SYMBOLS",
    "favor_profile_enable", "favor_profile_reset", "favor_profile_read", "favor_profile_slots",
    "favor_profile_name", "favor_device_error", "favor_attn_bidir_noalloc",
    "favor_kv_state", "favor_attn_from_state", "favor_attn_causal_step",
    "favor_attn_bidir_backward", "favor_attn_causal_backward",
    "favor_attn_causal_gated", "favor_attn_causal_step_gated", "favor_set_relpos",
    "favor_check_bounded_wait", "FAVOR_WAIT_CHECK_CODE",
]

FAVOR_OK, FAVOR_ERR_INVALID_ARG, FAVOR_ERR_UNSUPPORTED, FAVOR_ERR_NOMEM, FAVOR_ERR_CUDA = range(5)
FAVOR_KERNEL_SOFTMAX_POS, FAVOR_KERNEL_RELU, FAVOR_KERNEL_SOFTMAX_HYP, FAVOR_KERNEL_SOFTMAX_TRIG = 0, 1, 2, 3
FAVOR_DTYPE_F32, FAVOR_DTYPE_BF16 = 0, 1
KIND_CODES = {"softmax_pos": FAVOR_KERNEL_SOFTMAX_POS, "relu": FAVOR_KERNEL_RELU,
              "softmax_hyp": FAVOR_KERNEL_SOFTMAX_HYP, "softmax_trig": FAVOR_KERNEL_SOFTMAX_TRIG}
DTYPE_CODES = {"f32": FAVOR_DTYPE_F32, "bf16": FAVOR_DTYPE_BF16}

EXPORTED_SYMBOLS = ("favor_create", "favor_feature_map", "favor_attn_bidir", "favor_attn_causal",
                    "favor_destroy", "favor_status_str", "favor_last_error", "favor_launch_count",
                    "favor_profile_enable", "favor_profile_reset", "favor_profile_read", "favor_profile_slots",
                    "favor_profile_name", "favor_device_error", "favor_attn_bidir_noalloc",
                    "favor_kv_state", "favor_attn_from_state", "favor_attn_causal_step",
                    "favor_attn_bidir_backward", "favor_attn_causal_backward",
                    "favor_attn_causal_gated", "favor_attn_causal_step_gated", "favor_set_relpos",
                    "favor_check_bounded_wait")

_HERE = os.path.dirname(os.path.abspath(__file__))


def lib_path() -> str:
    return os.path.join(_HERE, "_lib", "libfavor.so")


class FavorLibraryMissing(RuntimeError):
    pass


class FavorError(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        super().__init__(f"{fn} -> {favor_status_str(status)}: {msg}")
        self.status = status


_LIB = None


def lib() -> ctypes.CDLL:
    """Load libfavor.so once; raise if it is missing."""
    global _LIB
    if _LIB is None:
        p = lib_path()
        if not os.path.exists(p):
            raise FavorLibraryMissing(f"{p} is not built; run random_feature_gb300.build.build() first")
        L = ctypes.CDLL(p)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.favor_create.argtypes = [ctypes.POINTER(vp), i, i, i, i, i, i, ctypes.POINTER(ctypes.c_float), f, i, i]
        L.favor_feature_map.argtypes = [vp, vp, vp, i, i, vp]
        L.favor_attn_bidir.argtypes = [vp, vp, vp, vp, vp, i, i, vp]
        L.favor_attn_causal.argtypes = [vp, vp, vp, vp, vp, i, i, vp]
        L.favor_destroy.argtypes = [vp]
        for fn in ("favor_create", "favor_feature_map", "favor_attn_bidir", "favor_attn_causal", "favor_destroy"):
            getattr(L, fn).restype = ctypes.c_int
        L.favor_status_str.argtypes = [i]
        L.favor_status_str.restype = ctypes.c_char_p
        L.favor_last_error.argtypes = []
        L.favor_last_error.restype = ctypes.c_char_p
        L.favor_launch_count.argtypes = []
        L.favor_launch_count.restype = ctypes.c_ulonglong
        L.favor_profile_enable.argtypes = [vp, i]
        L.favor_profile_reset.argtypes = [vp]
        L.favor_profile_read.argtypes = [vp, i, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_ulonglong)]
        for fn in ("favor_profile_enable", "favor_profile_reset", "favor_profile_read"):
            getattr(L, fn).restype = ctypes.c_int
        L.favor_profile_slots.argtypes = []
        L.favor_profile_slots.restype = i
        L.favor_profile_name.argtypes = [i]
        L.favor_profile_name.restype = ctypes.c_char_p
        L.favor_device_error.argtypes = [vp, ctypes.POINTER(i)]
        L.favor_device_error.restype = ctypes.c_int
        L.favor_attn_bidir_noalloc.argtypes = [vp, i, i, i, i, i, i, f, vp, vp, vp, vp, i, i, vp]
        L.favor_attn_bidir_noalloc.restype = ctypes.c_int
        L.favor_kv_state.argtypes = [vp, vp, vp, vp, i, i, vp]
        L.favor_attn_from_state.argtypes = [vp, vp, vp, vp, i, i, vp]
        L.favor_attn_causal_step.argtypes = [vp, vp, vp, vp, vp, vp, i, i, vp]
        for fn in ("favor_attn_bidir_backward", "favor_attn_causal_backward"):
            getattr(L, fn).argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, vp]
        L.favor_attn_causal_gated.argtypes = [vp, vp, vp, vp, vp, vp, i, i, vp]
        L.favor_attn_causal_step_gated.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, vp]
        L.favor_set_relpos.argtypes = [vp, vp, vp]
        L.favor_check_bounded_wait.argtypes = [vp, i, vp]
        L.favor_check_bounded_wait.restype = ctypes.c_int
        for fn in ("favor_kv_state", "favor_attn_from_state", "favor_attn_causal_step",
                   "favor_attn_bidir_backward", "favor_attn_causal_backward", "favor_attn_causal_gated",
                   "favor_attn_causal_step_gated", "favor_set_relpos"):
            getattr(L, fn).restype = ctypes.c_int
        _LIB = L
    return _LIB


def favor_status_str(status: int) -> str:
    return lib().favor_status_str(int(status)).decode()


def favor_last_error() -> str:
    return lib().favor_last_error().decode()


def favor_launch_count() -> int:
    return int(lib().favor_launch_count())


def _check(status: int, fn: str) -> None:
    if status != FAVOR_OK:
        raise FavorError(status, fn, favor_last_error())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream, like):
    if stream is None:
        import torch
        dev = like.device if hasattr(like, "device") else None
        return torch.cuda.current_stream(dev).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def favor_create(H, m, d, dv, kind, dtype, omega, data_scale, max_B, max_L) -> int:
    """Create a handle; ``omega`` is a host float32 array [H, m, d] ([H, m/2, d] for the
    hyperbolic and trigonometric kinds).  Returns the handle (int)."""
    kind = KIND_CODES.get(kind, kind)
    dtype = DTYPE_CODES.get(dtype, dtype)
    om = np.ascontiguousarray(omega, dtype=np.float32)
    rows = m // 2 if kind in (FAVOR_KERNEL_SOFTMAX_HYP, FAVOR_KERNEL_SOFTMAX_TRIG) else m
    if om.shape != (H, rows, d):
        raise ValueError(f"omega must have shape {(H, rows, d)}, got {om.shape}")
    h = ctypes.c_void_p()
    st = lib().favor_create(ctypes.byref(h), int(H), int(m), int(d), int(dv), int(kind), int(dtype),
                            om.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), float(data_scale),
                            int(max_B), int(max_L))
    _check(st, "favor_create")
    return h.value


def favor_feature_map(h, x, phi, B, L, stream=None) -> None:
    _check(lib().favor_feature_map(h, _ptr(x), _ptr(phi), int(B), int(L), _stream(stream, x)), "favor_feature_map")


def favor_attn_bidir(h, q, k, v, out, B, L, stream=None) -> None:
    _check(lib().favor_attn_bidir(h, _ptr(q), _ptr(k), _ptr(v), _ptr(out), int(B), int(L), _stream(stream, q)),
           "favor_attn_bidir")


def favor_attn_causal(h, q, k, v, out, B, L, stream=None) -> None:
    _check(lib().favor_attn_causal(h, _ptr(q), _ptr(k), _ptr(v), _ptr(out), int(B), int(L), _stream(stream, q)),
           "favor_attn_causal")


def favor_attn_bidir_noalloc(omega, H, m, d, dv, kind, dtype, data_scale, q, k, v, out, B, L,
                             stream=None) -> None:
    """Handle-free bidirectional call on the library's fixed device scratch; ``omega`` is a DEVICE
    float32 [H, m, d] tensor or address."""
    kind = KIND_CODES.get(kind, kind)
    dtype = DTYPE_CODES.get(dtype, dtype)
    _check(lib().favor_attn_bidir_noalloc(_ptr(omega), int(H), int(m), int(d), int(dv), int(kind), int(dtype),
                                          float(data_scale), _ptr(q), _ptr(k), _ptr(v), _ptr(out), int(B), int(L),
                                          _stream(stream, q)), "favor_attn_bidir_noalloc")


def favor_kv_state(h, k, v, state, B, L, stream=None) -> None:
    _check(lib().favor_kv_state(h, _ptr(k), _ptr(v), _ptr(state), int(B), int(L), _stream(stream, k)), "favor_kv_state")


def favor_attn_from_state(h, q, state, out, B, L, stream=None) -> None:
    _check(lib().favor_attn_from_state(h, _ptr(q), _ptr(state), _ptr(out), int(B), int(L), _stream(stream, q)),
           "favor_attn_from_state")


def favor_attn_causal_step(h, q, k, v, out, state, B, T, stream=None) -> None:
    _check(lib().favor_attn_causal_step(h, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(state), int(B), int(T),
                                        _stream(stream, q)), "favor_attn_causal_step")


def favor_attn_bidir_backward(h, q, k, v, dout, dq, dk, dv, B, L, stream=None) -> None:
    _check(lib().favor_attn_bidir_backward(h, _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                           int(B), int(L), _stream(stream, q)), "favor_attn_bidir_backward")


def favor_attn_causal_backward(h, q, k, v, dout, dq, dk, dv, B, L, stream=None) -> None:
    _check(lib().favor_attn_causal_backward(h, _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                            int(B), int(L), _stream(stream, q)), "favor_attn_causal_backward")


def favor_attn_causal_gated(h, q, k, v, gate, out, B, L, stream=None) -> None:
    _check(lib().favor_attn_causal_gated(h, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(out), int(B), int(L),
                                         _stream(stream, q)), "favor_attn_causal_gated")


def favor_attn_causal_step_gated(h, q, k, v, gate, out, state, B, T, stream=None) -> None:
    _check(lib().favor_attn_causal_step_gated(h, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(out), _ptr(state),
                                              int(B), int(T), _stream(stream, q)), "favor_attn_causal_step_gated")


def favor_set_relpos(h, perm=None, r=None) -> None:
    """PermuteFormer setting: host int [H, m] permutations (or None) and host float [H] decays (or None)."""
    pa = None if perm is None else np.ascontiguousarray(perm, dtype=np.int32)
    ra = None if r is None else np.ascontiguousarray(r, dtype=np.float32)
    _check(lib().favor_set_relpos(h, None if pa is None else pa.ctypes.data, None if ra is None else ra.ctypes.data),
           "favor_set_relpos")


def favor_destroy(h) -> None:
    _check(lib().favor_destroy(h), "favor_destroy")


def favor_profile_enable(h, enable=True) -> None:
    _check(lib().favor_profile_enable(h, 1 if enable else 0), "favor_profile_enable")


def favor_profile_reset(h) -> None:
    _check(lib().favor_profile_reset(h), "favor_profile_reset")


def favor_profile_read(h, slot):
    """(total device ms, launches) recorded for one kernel slot (synchronises)."""
    ms = ctypes.c_double()
    n = ctypes.c_ulonglong()
    _check(lib().favor_profile_read(h, int(slot), ctypes.byref(ms), ctypes.byref(n)), "favor_profile_read")
    return ms.value, n.value


def favor_device_error(h) -> int:
    """Synchronise and return the handle's device error word (0 = no bounded wait gave up)."""
    code = ctypes.c_int()
    _check(lib().favor_device_error(h, ctypes.byref(code)), "favor_device_error")
    return code.value


FAVOR_WAIT_CHECK_CODE = 901


def favor_check_bounded_wait(h, limit_cycles: int, stream=None) -> None:
    """Enqueue the bounded-wait check kernel (a wait that nothing completes gives
    up after limit_cycles cycles and writes FAVOR_WAIT_CHECK_CODE to the
    handle's device error word)."""
    _check(lib().favor_check_bounded_wait(h, int(limit_cycles), _stream(stream, None)), "favor_check_bounded_wait")


def favor_profile_slots() -> int:
    return int(lib().favor_profile_slots())


def favor_profile_name(slot) -> str:
    return lib().favor_profile_name(int(slot)).decode()


class Favor:
    """Owns one handle; checks torch tensor shapes/dtypes before calling the C ABI."""

    def __init__(self, H, m, d, dv, kind, dtype, omega, data_scale, max_B, max_L):
        self.H, self.m, self.d, self.dv = H, m, d, dv
        self.kind, self.dtype = kind, dtype
        self.max_B, self.max_L = max_B, max_L
        self.handle = favor_create(H, m, d, dv, kind, dtype, omega, data_scale, max_B, max_L)

    def _tdtype(self):
        import torch
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def _chk(self, t, B, L, w, name):
        if tuple(t.shape) != (B, self.H, L, w) or t.dtype != self._tdtype() or not t.is_cuda \
                or not t.is_contiguous():
            raise ValueError(f"{name}: expected contiguous CUDA {self._tdtype()} [{B},{self.H},{L},{w}], "
                             f"got {t.dtype} {tuple(t.shape)} on {t.device}")

    def _new(self, like, B, L, w, out):
        import torch
        if out is None:
            out = torch.empty((B, self.H, L, w), dtype=self._tdtype(), device=like.device)
        self._chk(out, B, L, w, "out")
        return out

    def feature_map(self, x, out=None, stream=None):
        B, _, L, _ = x.shape
        self._chk(x, B, L, self.d, "x")
        out = self._new(x, B, L, self.m, out)
        favor_feature_map(self.handle, x, out, B, L, stream)
        return out

    def attn(self, q, k, v, causal=False, out=None, stream=None):
        B, _, L, _ = q.shape
        self._chk(q, B, L, self.d, "q")
        self._chk(k, B, L, self.d, "k")
        self._chk(v, B, L, self.dv, "v")
        out = self._new(q, B, L, self.dv, out)
        (favor_attn_causal if causal else favor_attn_bidir)(self.handle, q, k, v, out, B, L, stream)
        return out

    def attn_backward(self, q, k, v, dout, causal=False, grads=None, stream=None):
        """(dq, dk, dv) of attn(q, k, v, causal) for the upstream gradient dout.
        ``grads`` may give the three output tensors."""
        B, _, L, _ = q.shape
        for t, w, name in ((q, self.d, "q"), (k, self.d, "k"), (v, self.dv, "v"), (dout, self.dv, "dout")):
            self._chk(t, B, L, w, name)
        if grads is None:
            grads = (self._new(q, B, L, self.d, None), self._new(q, B, L, self.d, None),
                     self._new(q, B, L, self.dv, None))
        dq, dk, dv = grads
        self._chk(dq, B, L, self.d, "dq")
        self._chk(dk, B, L, self.d, "dk")
        self._chk(dv, B, L, self.dv, "dv")
        fn = favor_attn_causal_backward if causal else favor_attn_bidir_backward
        fn(self.handle, q, k, v, dout, dq, dk, dv, B, L, stream)
        return dq, dk, dv

    def attn_causal_gated(self, q, k, v, gate, out=None, stream=None):
        """RFA-Gate causal attention; gate is a CUDA float32 [B, H, L] tensor."""
        import torch
        B, _, L, _ = q.shape
        self._chk(q, B, L, self.d, "q")
        self._chk(k, B, L, self.d, "k")
        self._chk(v, B, L, self.dv, "v")
        if tuple(gate.shape) != (B, self.H, L) or gate.dtype != torch.float32 or not gate.is_cuda \
                or not gate.is_contiguous():
            raise ValueError(f"gate: expected contiguous CUDA float32 [{B},{self.H},{L}]")
        out = self._new(q, B, L, self.dv, out)
        favor_attn_causal_gated(self.handle, q, k, v, gate, out, B, L, stream)
        return out

    def causal_step_gated(self, q, k, v, gate, state, out=None, stream=None):
        import torch
        B, _, T, _ = q.shape
        self._chk(q, B, T, self.d, "q")
        self._chk(k, B, T, self.d, "k")
        self._chk(v, B, T, self.dv, "v")
        self._chk_state(state, B)
        if tuple(gate.shape) != (B, self.H, T) or gate.dtype != torch.float32 or not gate.is_cuda \
                or not gate.is_contiguous():
            raise ValueError(f"gate: expected contiguous CUDA float32 [{B},{self.H},{T}]")
        out = self._new(q, B, T, self.dv, out)
        favor_attn_causal_step_gated(self.handle, q, k, v, gate, out, state, B, T, stream)
        return out

    def set_relpos(self, perm=None, r=None):
        favor_set_relpos(self.handle, perm, r)

    def new_state(self, B):
        """A zero (empty) state [B, H, m, dv+1] float32 on the current CUDA device."""
        import torch
        return torch.zeros((B, self.H, self.m, self.dv + 1), dtype=torch.float32, device="cuda")

    def _chk_state(self, state, B):
        import torch
        if tuple(state.shape) != (B, self.H, self.m, self.dv + 1) or state.dtype != torch.float32 \
                or not state.is_cuda or not state.is_contiguous():
            raise ValueError(f"state: expected contiguous CUDA float32 [{B},{self.H},{self.m},{self.dv + 1}], "
                             f"got {state.dtype} {tuple(state.shape)} on {state.device}")

    def kv_state(self, k, v, state=None, stream=None):
        """state += summary of (k, v); a new zero state if none is given.  Returns the state."""
        B, _, L, _ = k.shape
        self._chk(k, B, L, self.d, "k")
        self._chk(v, B, L, self.dv, "v")
        if state is None:
            state = self.new_state(B)
        self._chk_state(state, B)
        favor_kv_state(self.handle, k, v, state, B, L, stream)
        return state

    def attn_from_state(self, q, state, out=None, stream=None):
        B, _, L, _ = q.shape
        self._chk(q, B, L, self.d, "q")
        self._chk_state(state, B)
        out = self._new(q, B, L, self.dv, out)
        favor_attn_from_state(self.handle, q, state, out, B, L, stream)
        return out

    def causal_step(self, q, k, v, state, out=None, stream=None):
        """Causal attention of T new tokens continuing from state (updated in place)."""
        B, _, T, _ = q.shape
        self._chk(q, B, T, self.d, "q")
        self._chk(k, B, T, self.d, "k")
        self._chk(v, B, T, self.dv, "v")
        self._chk_state(state, B)
        out = self._new(q, B, T, self.dv, out)
        favor_attn_causal_step(self.handle, q, k, v, out, state, B, T, stream)
        return out

    def close(self):
        if self.handle:
            favor_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
