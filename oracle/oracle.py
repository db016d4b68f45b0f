"""Python face of the lrscan oracle -- TEST INFRASTRUCTURE ONLY.

The oracle is the plain C statement of the diagonal linear-recurrence scan in
``lrscan_oracle.c`` (forward h_t = a_t*h_{t-1} + b_t and its reverse-mode
gradient, as defined by triton_training_scan.py, _real_forward and
_real_backward).  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It never touches the
CUDA library, and the CUDA library never touches it.

Arrays are numpy, contiguous, shaped [B, T, D] (``last`` is [B, D]):
  * ``"f32"``  -- float32 storage, fp32 state, fused multiply-add steps;
  * ``"bf16"`` -- uint16 arrays holding bf16 bit patterns, fp32 state,
                  round-to-nearest-even on every store;
  * ``"f64"``  -- float64 storage and state.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lrscan_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liblrscan_oracle.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None

_I64 = ctypes.c_int64
_P = ctypes.c_void_p


def compile_library(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc; returns the path of the shared object."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build() -> str:
    """Build the oracle if the shared object is missing or older than its source."""
    if (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        compile_library()
    return _LIB_PATH


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    for name in ("lro_fwd_f32", "lro_fwd_bf16", "lro_fwd_f64"):
        getattr(lib, name).argtypes = [_P, _P, _P, _P, _I64, _I64, _I64]
        getattr(lib, name).restype = ctypes.c_int
    for name in ("lro_bwd_f32", "lro_bwd_bf16", "lro_bwd_f64"):
        getattr(lib, name).argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64]
        getattr(lib, name).restype = ctypes.c_int
    for name in ("lro_chunk_fwd_f32", "lro_chunk_fwd_f64"):
        getattr(lib, name).argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I64]
        getattr(lib, name).restype = ctypes.c_int
    for name in ("lro_chunk_bwd_f32", "lro_chunk_bwd_f64"):
        getattr(lib, name).argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64]
        getattr(lib, name).restype = ctypes.c_int
    for name in ("lro_fwd_state_f32", "lro_fwd_state_bf16", "lro_fwd_state_f64"):
        getattr(lib, name).argtypes = [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64]
        getattr(lib, name).restype = ctypes.c_int
    for name in ("lro_bwd_state_f32", "lro_bwd_state_bf16", "lro_bwd_state_f64"):
        getattr(lib, name).argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64]
        getattr(lib, name).restype = ctypes.c_int
    for name in ("lro_cfwd_f32", "lro_cfwd_bf16", "lro_cfwd_f64"):
        getattr(lib, name).argtypes = [_P] * 8 + [_I64, _I64, _I64]
        getattr(lib, name).restype = ctypes.c_int
    for name in ("lro_cbwd_f32", "lro_cbwd_bf16", "lro_cbwd_f64"):
        getattr(lib, name).argtypes = [_P] * 10 + [_I64, _I64, _I64]
        getattr(lib, name).restype = ctypes.c_int
    for name in ("lro_cfwd_state_f32", "lro_cfwd_state_bf16", "lro_cfwd_state_f64"):
        getattr(lib, name).argtypes = [_P] * 11 + [_I64, _I64, _I64]
        getattr(lib, name).restype = ctypes.c_int
    for name in ("lro_cbwd_state_f32", "lro_cbwd_state_bf16", "lro_cbwd_state_f64"):
        getattr(lib, name).argtypes = [_P] * 17 + [_I64, _I64, _I64]
        getattr(lib, name).restype = ctypes.c_int
    for name in ("lro_gated_fwd_f32", "lro_gated_fwd_bf16", "lro_gated_fwd_f64"):
        getattr(lib, name).argtypes = [_P] * 5 + [_I64, _I64, _I64]
        getattr(lib, name).restype = ctypes.c_int
    for name in ("lro_gated_bwd_f32", "lro_gated_bwd_bf16", "lro_gated_bwd_f64"):
        getattr(lib, name).argtypes = [_P] * 7 + [_I64, _I64, _I64]
        getattr(lib, name).restype = ctypes.c_int
    lib.lro_f32_to_bf16_array.argtypes = [_P, _P, _I64]
    lib.lro_bf16_to_f32_array.argtypes = [_P, _P, _I64]
    lib.lro_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.lro_f32_to_bf16.restype = ctypes.c_uint16
    lib.lro_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.lro_bf16_to_f32.restype = ctypes.c_float
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library.

    ``path`` selects another build of the same source, which the mutation
    tests use to check that the pins catch planted mistakes.
    """
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


_NP = {"f32": np.float32, "bf16": np.uint16, "f64": np.float64}
_LAST = {"f32": np.float32, "bf16": np.float32, "f64": np.float64}


def _c(x: np.ndarray, dtype: str) -> np.ndarray:
    want = _NP[dtype]
    if x.dtype != want:
        raise TypeError(f"oracle {dtype} expects {np.dtype(want).name}, got {x.dtype}")
    if x.ndim != 3:
        raise ValueError("oracle expects [B, T, D] arrays")
    return np.ascontiguousarray(x)


def _ptr(x: np.ndarray) -> int:
    return x.ctypes.data


class Oracle:
    """Bound view of one build of the oracle library."""

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else load()

    def fwd(self, a: np.ndarray, b: np.ndarray, dtype: str = "f32"):
        """Sequential forward scan; returns ``(out, last)``."""
        a, b = _c(a, dtype), _c(b, dtype)
        if a.shape != b.shape:
            raise ValueError("a and b must have the same [B, T, D] shape")
        B, T, D = a.shape
        out = np.empty_like(a)
        last = np.empty((B, D), dtype=_LAST[dtype])
        rc = getattr(self.lib, f"lro_fwd_{dtype}")(_ptr(a), _ptr(b), _ptr(out), _ptr(last), B, T, D)
        if rc:
            raise RuntimeError(f"oracle forward failed ({rc})")
        return out, last

    def bwd(self, a: np.ndarray, out: np.ndarray, grad_out: np.ndarray, dtype: str = "f32"):
        """Sequential reverse scan; returns ``(grad_a, grad_b)``."""
        a, out, grad_out = _c(a, dtype), _c(out, dtype), _c(grad_out, dtype)
        if not (a.shape == out.shape == grad_out.shape):
            raise ValueError("a, out and grad_out must have the same [B, T, D] shape")
        B, T, D = a.shape
        ga, gb = np.empty_like(a), np.empty_like(a)
        rc = getattr(self.lib, f"lro_bwd_{dtype}")(_ptr(a), _ptr(out), _ptr(grad_out),
                                                    _ptr(ga), _ptr(gb), B, T, D)
        if rc:
            raise RuntimeError(f"oracle backward failed ({rc})")
        return ga, gb

    def chunk_fwd(self, a: np.ndarray, b: np.ndarray, chunk: int, dtype: str = "f64"):
        """Two-level (summary, serial prefix, replay) forward; ``(out, last)``."""
        a, b = _c(a, dtype), _c(b, dtype)
        B, T, D = a.shape
        out = np.empty_like(a)
        last = np.empty((B, D), dtype=_LAST[dtype])
        rc = getattr(self.lib, f"lro_chunk_fwd_{dtype}")(_ptr(a), _ptr(b), _ptr(out), _ptr(last),
                                                          B, T, D, chunk)
        if rc:
            raise RuntimeError(f"oracle chunk forward failed ({rc})")
        return out, last

    def chunk_bwd(self, a: np.ndarray, out: np.ndarray, grad_out: np.ndarray, chunk: int,
                  dtype: str = "f64"):
        """Two-level reverse scan; ``(grad_a, grad_b)``."""
        a, out, grad_out = _c(a, dtype), _c(out, dtype), _c(grad_out, dtype)
        B, T, D = a.shape
        ga, gb = np.empty_like(a), np.empty_like(a)
        rc = getattr(self.lib, f"lro_chunk_bwd_{dtype}")(_ptr(a), _ptr(out), _ptr(grad_out),
                                                          _ptr(ga), _ptr(gb), B, T, D, chunk)
        if rc:
            raise RuntimeError(f"oracle chunk backward failed ({rc})")
        return ga, gb

    def _state(self, x, dtype, shape, what):
        if x is None:
            return None
        want = _LAST[dtype]
        if x.dtype != want or tuple(x.shape) != tuple(shape):
            raise TypeError(f"oracle {dtype} {what} must be {np.dtype(want).name} {tuple(shape)}")
        return np.ascontiguousarray(x)

    @staticmethod
    def _seg(seg, B, T):
        if seg is None:
            return None
        if seg.dtype != np.int32 or seg.shape != (B, T):
            raise TypeError("segment_pos must be int32 [B, T]")
        return np.ascontiguousarray(seg)

    def fwd_state(self, a, b, dtype="f32", h0=None, segment_pos=None):
        """Forward scan from the initial state h0 with segment resets
        (steps where segment_pos == 0 ignore the previous state); ``(out, last)``."""
        a, b = _c(a, dtype), _c(b, dtype)
        if a.shape != b.shape:
            raise ValueError("a and b must have the same [B, T, D] shape")
        B, T, D = a.shape
        h0 = self._state(h0, dtype, (B, D), "h0")
        seg = self._seg(segment_pos, B, T)
        out = np.empty_like(a)
        last = np.empty((B, D), dtype=_LAST[dtype])
        rc = getattr(self.lib, f"lro_fwd_state_{dtype}")(
            _ptr(a), _ptr(b), _ptr(out), _ptr(last), None if h0 is None else _ptr(h0),
            None if seg is None else _ptr(seg), B, T, D)
        if rc:
            raise RuntimeError(f"oracle state forward failed ({rc})")
        return out, last

    def bwd_state(self, a, out, grad_out, dtype="f32", h0=None, segment_pos=None, grad_last=None):
        """Reverse scan of :meth:`fwd_state`; ``(grad_a, grad_b, grad_h0)``."""
        a, out, grad_out = _c(a, dtype), _c(out, dtype), _c(grad_out, dtype)
        if not (a.shape == out.shape == grad_out.shape):
            raise ValueError("a, out and grad_out must have the same [B, T, D] shape")
        B, T, D = a.shape
        h0 = self._state(h0, dtype, (B, D), "h0")
        gl = self._state(grad_last, dtype, (B, D), "grad_last")
        seg = self._seg(segment_pos, B, T)
        ga, gb = np.empty_like(a), np.empty_like(a)
        gh0 = np.empty((B, D), dtype=_LAST[dtype])
        rc = getattr(self.lib, f"lro_bwd_state_{dtype}")(
            _ptr(a), _ptr(out), _ptr(grad_out), None if h0 is None else _ptr(h0),
            None if seg is None else _ptr(seg), None if gl is None else _ptr(gl),
            _ptr(ga), _ptr(gb), _ptr(gh0), B, T, D)
        if rc:
            raise RuntimeError(f"oracle state backward failed ({rc})")
        return ga, gb, gh0

    def cfwd(self, ar, ai, br, bi, dtype="f32"):
        """Complex forward scan on re/im planes; ``(out_r, out_i, last_r, last_i)``."""
        xs = [_c(x, dtype) for x in (ar, ai, br, bi)]
        if any(x.shape != xs[0].shape for x in xs):
            raise ValueError("ar, ai, br, bi must have the same [B, T, D] shape")
        B, T, D = xs[0].shape
        out_r, out_i = np.empty_like(xs[0]), np.empty_like(xs[0])
        last_r = np.empty((B, D), dtype=_LAST[dtype])
        last_i = np.empty((B, D), dtype=_LAST[dtype])
        rc = getattr(self.lib, f"lro_cfwd_{dtype}")(*[_ptr(x) for x in xs], _ptr(out_r), _ptr(out_i),
                                                     _ptr(last_r), _ptr(last_i), B, T, D)
        if rc:
            raise RuntimeError(f"oracle complex forward failed ({rc})")
        return out_r, out_i, last_r, last_i

    def cbwd(self, ar, ai, out_r, out_i, go_r, go_i, dtype="f32"):
        """Complex reverse scan; ``(grad_ar, grad_ai, grad_br, grad_bi)``."""
        xs = [_c(x, dtype) for x in (ar, ai, out_r, out_i, go_r, go_i)]
        if any(x.shape != xs[0].shape for x in xs):
            raise ValueError("complex backward inputs must have the same [B, T, D] shape")
        B, T, D = xs[0].shape
        gs = [np.empty_like(xs[0]) for _ in range(4)]
        rc = getattr(self.lib, f"lro_cbwd_{dtype}")(*[_ptr(x) for x in xs], *[_ptr(g) for g in gs], B, T, D)
        if rc:
            raise RuntimeError(f"oracle complex backward failed ({rc})")
        return tuple(gs)

    def cfwd_state(self, ar, ai, br, bi, dtype="f32", h0=None, segment_pos=None):
        """Complex forward scan from the initial state h0 = (re, im) with segment
        resets; ``(out_r, out_i, last_r, last_i)``."""
        xs = [_c(x, dtype) for x in (ar, ai, br, bi)]
        if any(x.shape != xs[0].shape for x in xs):
            raise ValueError("ar, ai, br, bi must have the same [B, T, D] shape")
        B, T, D = xs[0].shape
        h0r, h0i = (None, None) if h0 is None else (self._state(h0[0], dtype, (B, D), "h0_r"),
                                                    self._state(h0[1], dtype, (B, D), "h0_i"))
        seg = self._seg(segment_pos, B, T)
        out_r, out_i = np.empty_like(xs[0]), np.empty_like(xs[0])
        last_r = np.empty((B, D), dtype=_LAST[dtype])
        last_i = np.empty((B, D), dtype=_LAST[dtype])
        opt = lambda x: None if x is None else _ptr(x)  # noqa: E731
        rc = getattr(self.lib, f"lro_cfwd_state_{dtype}")(*[_ptr(x) for x in xs], _ptr(out_r), _ptr(out_i),
                                                           _ptr(last_r), _ptr(last_i), opt(h0r), opt(h0i), opt(seg),
                                                           B, T, D)
        if rc:
            raise RuntimeError(f"oracle complex state forward failed ({rc})")
        return out_r, out_i, last_r, last_i

    def cbwd_state(self, ar, ai, out_r, out_i, go_r, go_i, dtype="f32", h0=None, segment_pos=None,
                   grad_last=None):
        """Reverse scan of :meth:`cfwd_state`; ``(grad_ar, grad_ai, grad_br,
        grad_bi, grad_h0_r, grad_h0_i)``."""
        xs = [_c(x, dtype) for x in (ar, ai, out_r, out_i, go_r, go_i)]
        if any(x.shape != xs[0].shape for x in xs):
            raise ValueError("complex backward inputs must have the same [B, T, D] shape")
        B, T, D = xs[0].shape
        h0r, h0i = (None, None) if h0 is None else (self._state(h0[0], dtype, (B, D), "h0_r"),
                                                    self._state(h0[1], dtype, (B, D), "h0_i"))
        glr, gli = (None, None) if grad_last is None else (self._state(grad_last[0], dtype, (B, D), "grad_last_r"),
                                                           self._state(grad_last[1], dtype, (B, D), "grad_last_i"))
        seg = self._seg(segment_pos, B, T)
        gs = [np.empty_like(xs[0]) for _ in range(4)]
        gh0 = [np.empty((B, D), dtype=_LAST[dtype]) for _ in range(2)]
        opt = lambda x: None if x is None else _ptr(x)  # noqa: E731
        rc = getattr(self.lib, f"lro_cbwd_state_{dtype}")(*[_ptr(x) for x in xs], opt(h0r), opt(h0i), opt(seg),
                                                           opt(glr), opt(gli), *[_ptr(g) for g in gs],
                                                           _ptr(gh0[0]), _ptr(gh0[1]), B, T, D)
        if rc:
            raise RuntimeError(f"oracle complex state backward failed ({rc})")
        return (*gs, *gh0)

    def _gated_params(self, eta, nu_log, dtype, B, T, D):
        want = _LAST[dtype]
        eta = np.ascontiguousarray(eta)
        nu_log = np.ascontiguousarray(nu_log)
        if eta.dtype != want or eta.shape != (B, T) or nu_log.dtype != want or nu_log.shape != (D,):
            raise TypeError(f"eta must be {np.dtype(want).name} [B, T] and nu_log {np.dtype(want).name} [D]")
        return eta, nu_log

    def gated_fwd(self, eta, nu_log, b, dtype="f32"):
        """Scan with the decay generated as exp(-exp(nu_log_d) * exp(eta_t)); ``(out, last)``."""
        b = _c(b, dtype)
        B, T, D = b.shape
        eta, nu_log = self._gated_params(eta, nu_log, dtype, B, T, D)
        out = np.empty_like(b)
        last = np.empty((B, D), dtype=_LAST[dtype])
        rc = getattr(self.lib, f"lro_gated_fwd_{dtype}")(_ptr(eta), _ptr(nu_log), _ptr(b), _ptr(out), _ptr(last),
                                                          B, T, D)
        if rc:
            raise RuntimeError(f"oracle gated forward failed ({rc})")
        return out, last

    def gated_bwd(self, eta, nu_log, out, grad_out, dtype="f32"):
        """Reverse of :meth:`gated_fwd`; ``(grad_b, grad_eta, grad_nu_log)``."""
        out, grad_out = _c(out, dtype), _c(grad_out, dtype)
        B, T, D = out.shape
        eta, nu_log = self._gated_params(eta, nu_log, dtype, B, T, D)
        gb = np.empty_like(out)
        geta = np.empty((B, T), dtype=_LAST[dtype])
        gnu = np.empty((D,), dtype=_LAST[dtype])
        rc = getattr(self.lib, f"lro_gated_bwd_{dtype}")(_ptr(eta), _ptr(nu_log), _ptr(out), _ptr(grad_out),
                                                          _ptr(gb), _ptr(geta), _ptr(gnu), B, T, D)
        if rc:
            raise RuntimeError(f"oracle gated backward failed ({rc})")
        return gb, geta, gnu

    def f32_to_bf16(self, x: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty(x.shape, dtype=np.uint16)
        self.lib.lro_f32_to_bf16_array(_ptr(x), _ptr(y), x.size)
        return y

    def bf16_to_f32(self, x: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.uint16)
        y = np.empty(x.shape, dtype=np.float32)
        self.lib.lro_bf16_to_f32_array(_ptr(x), _ptr(y), x.size)
        return y


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
