"""Python binding of liblrscan.so (argument marshalling only).

Every function here checks tensors, picks the stream and hands raw device
pointers to the C ABI declared in ``include/lrscan.h``; all arithmetic runs in
the library's CUDA kernels.  PyTorch supplies device memory and streams.

If the library has not been built (``__graft_entry__.build()`` or
``python -m linear_recurrence_scan_lrscan_gb300.build``) every call raises
``LrscanUnavailable``: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

LRSCAN_OK = 0
LRSCAN_EINVAL = -1
LRSCAN_EDTYPE = -2
LRSCAN_ECUDA = -3
LRSCAN_ENOMEM = -4
LRSCAN_ETIMEOUT = -5
LRSCAN_ENODEVICE = -6

F32, BF16 = 0, 1
PATHS = {"auto": 0, "seq": 1, "chunk": 2, "window": 3, "plain": 4, "stream": 5}
PATH_NAMES = {v: k for k, v in PATHS.items()}
_DTYPES = {torch.float32: F32, torch.bfloat16: BF16}

_I64 = ctypes.c_int64
_P = ctypes.c_void_p


class LrscanUnavailable(RuntimeError):
    """The CUDA library is missing or could not be loaded."""


class LrscanError(RuntimeError):
    def __init__(self, code: int, what: str):
        detail = ""
        try:
            detail = lib().lrscan_last_error().decode()
        except LrscanUnavailable:
            pass
        super().__init__(f"{what}: {strerror(code)} ({code})" + (f": {detail}" if detail else ""))
        self.code = code
        self.detail = detail


class Opts(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("chunk_len", ctypes.c_int), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("tile_variant", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("tile_variant", ctypes.c_int), ("lanes_per_cta", ctypes.c_int),
                ("rows_per_window", ctypes.c_int), ("subchunks", ctypes.c_int), ("stages", ctypes.c_int),
                ("ctas", ctypes.c_int), ("threads_per_cta", ctypes.c_int), ("smem_bytes", ctypes.c_int),
                ("kernels", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t), ("name", ctypes.c_char * 64),
                ("exact", ctypes.c_int)]

    def as_dict(self) -> dict:
        d = {k: getattr(self, k) for k, _ in self._fields_ if k != "name"}
        d["name"] = self.name.decode()
        d["path"] = PATH_NAMES.get(self.path, self.path)
        return d


class State(ctypes.Structure):
    _fields_ = [("h0", ctypes.c_void_p), ("segment_pos", ctypes.c_void_p), ("grad_last", ctypes.c_void_p),
                ("grad_h0", ctypes.c_void_p)]


class CState(ctypes.Structure):
    _fields_ = [("h0_r", ctypes.c_void_p), ("h0_i", ctypes.c_void_p), ("segment_pos", ctypes.c_void_p),
                ("grad_last_r", ctypes.c_void_p), ("grad_last_i", ctypes.c_void_p), ("grad_h0_r", ctypes.c_void_p),
                ("grad_h0_i", ctypes.c_void_p)]


EXPORTS = {
    "lrscan_fwd": ([_P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int], ctypes.c_int),
    "lrscan_bwd": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int], ctypes.c_int),
    "lrscan_fwd_ex": ([_P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int, _P, ctypes.POINTER(Opts)], ctypes.c_int),
    "lrscan_bwd_ex": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int, _P, ctypes.POINTER(Opts)],
                      ctypes.c_int),
    "lrscan_fwd_host": ([_P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int, ctypes.POINTER(Opts)], ctypes.c_int),
    "lrscan_bwd_host": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int, ctypes.POINTER(Opts)],
                        ctypes.c_int),
    "lrscan_fwd_bwd_host": ([_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int, ctypes.POINTER(Opts)],
                            ctypes.c_int),
    "lrscan_fwd_state": ([_P, _P, _P, _P, ctypes.POINTER(State), _I64, _I64, _I64, ctypes.c_int, _P,
                          ctypes.POINTER(Opts)], ctypes.c_int),
    "lrscan_bwd_state": ([_P, _P, _P, _P, _P, ctypes.POINTER(State), _I64, _I64, _I64, ctypes.c_int, _P,
                          ctypes.POINTER(Opts)], ctypes.c_int),
    "lrscan_summary": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, _P], ctypes.c_int),
    "lrscan_compose_maps": ([_P, _I64, _I64, _P, _P, _I64, _I64, ctypes.c_int, _P], ctypes.c_int),
    "lrscan_cfwd": ([_P] * 8 + [_I64, _I64, _I64, ctypes.c_int, _P, ctypes.POINTER(Opts)], ctypes.c_int),
    "lrscan_cbwd": ([_P] * 10 + [_I64, _I64, _I64, ctypes.c_int, _P, ctypes.POINTER(Opts)], ctypes.c_int),
    "lrscan_cfwd_state": ([_P] * 8 + [ctypes.POINTER(CState), _I64, _I64, _I64, ctypes.c_int, _P,
                                     ctypes.POINTER(Opts)], ctypes.c_int),
    "lrscan_cbwd_state": ([_P] * 10 + [ctypes.POINTER(CState), _I64, _I64, _I64, ctypes.c_int, _P,
                                      ctypes.POINTER(Opts)], ctypes.c_int),
    "lrscan_plan_complex": ([_I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(Opts),
                             ctypes.POINTER(PlanInfo)], ctypes.c_int),
    "lrscan_plan_complex_state": ([_I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.POINTER(Opts), ctypes.POINTER(PlanInfo)], ctypes.c_int),
    "lrscan_fwd_gated": ([_P] * 5 + [_I64, _I64, _I64, ctypes.c_int, _P, ctypes.POINTER(Opts)], ctypes.c_int),
    "lrscan_bwd_gated": ([_P] * 7 + [_I64, _I64, _I64, ctypes.c_int, _P, ctypes.POINTER(Opts)], ctypes.c_int),
    "lrscan_gated_workspace_bytes": ([_I64, _I64, _I64], ctypes.c_size_t),
    "lrscan_plan_gated": ([_I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(Opts),
                           ctypes.POINTER(PlanInfo)], ctypes.c_int),
    "lrscan_set_stream": ([_P], ctypes.c_int),
    "lrscan_workspace_bytes": ([_I64, _I64, _I64, ctypes.c_int], ctypes.c_size_t),
    "lrscan_plan": ([_I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(Opts),
                     ctypes.POINTER(PlanInfo)], ctypes.c_int),
    "lrscan_plan_state": ([_I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(Opts),
                           ctypes.POINTER(PlanInfo)], ctypes.c_int),
    "lrscan_num_variants": ([ctypes.c_int, ctypes.c_int, ctypes.c_int], ctypes.c_int),
    "lrscan_sync_check": ([], ctypes.c_int),
    "lrscan_set_wait_timeout_ns": ([ctypes.c_uint64], ctypes.c_int),
    "lrscan_selftest_wait_timeout": ([ctypes.c_uint64], ctypes.c_int),
    "lrscan_strerror": ([ctypes.c_int], ctypes.c_char_p),
    "lrscan_version": ([], ctypes.c_int),
    "lrscan_last_error": ([], ctypes.c_char_p),
    "lrscan_fwd_chunk_noalloc": ([_P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, _P], ctypes.c_int),
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return os.environ.get("LRSCAN_LIBRARY", _build.LIB)


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises LrscanUnavailable if it is not built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise LrscanUnavailable(
                    f"liblrscan.so not found at {path}; build it with "
                    "`python -m linear_recurrence_scan_lrscan_gb300.build` (nvcc, sm_103a)")
            try:
                handle = ctypes.CDLL(path)
            except OSError as e:  # pragma: no cover - depends on the machine
                raise LrscanUnavailable(f"cannot load {path}: {e}") from e
            for name, (argtypes, restype) in EXPORTS.items():
                fn = getattr(handle, name)
                fn.argtypes = argtypes
                fn.restype = restype
            _lib = handle
        return _lib


def strerror(code: int) -> str:
    try:
        return lib().lrscan_strerror(code).decode()
    except LrscanUnavailable:
        return f"error {code}"


def _check(rc: int, what: str) -> None:
    if rc != LRSCAN_OK:
        raise LrscanError(rc, what)


def _opts(path, chunk_len, tile_variant, workspace) -> Opts | None:
    if path is None and chunk_len is None and tile_variant is None and workspace is None:
        return None
    o = Opts()
    o.path = PATHS[path] if isinstance(path, str) else int(path or 0)
    o.chunk_len = int(chunk_len or 0)
    o.tile_variant = int(tile_variant or 0)
    if workspace is not None:
        if not workspace.is_cuda:
            raise ValueError("workspace must be a CUDA tensor")
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    return o


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check_tensors(shape, dtype, device, **tensors):
    for name, t in tensors.items():
        if t is None:
            continue
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if not t.is_cuda:
            raise ValueError(f"{name} must be on a CUDA device")
        if t.device != device:
            raise ValueError(f"{name} is on {t.device}, expected {device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if name == "last":
            if t.dtype != torch.float32 or tuple(t.shape) != (shape[0], shape[2]):
                raise ValueError("last must be fp32 [B, D]")
            continue
        if t.dtype != dtype:
            raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {t.dtype}; lrscan takes float32 or bfloat16 storage")
    return _DTYPES[t.dtype]


def lrscan_fwd(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None,
               last: torch.Tensor | None = None, *, want_last: bool = True, path=None,
               chunk_len=None, tile_variant=None, workspace=None, stream=None):
    """Forward scan h_t = a_t*h_{t-1} + b_t over [B, T, D]; returns (out, last)."""
    if a.ndim != 3 or a.shape != b.shape:
        raise ValueError("lrscan expects matching [B, T, D] tensors")
    code = _dtype_code(a)
    B, T, D = a.shape
    if out is None:
        out = torch.empty_like(b)
    if last is None and want_last:
        last = torch.empty((B, D), device=a.device, dtype=torch.float32)
    _check_tensors(a.shape, a.dtype, a.device, a=a, b=b, out=out, last=last)
    with torch.cuda.device(a.device):
        o = _opts(path, chunk_len, tile_variant, workspace)
        rc = lib().lrscan_fwd_ex(a.data_ptr(), b.data_ptr(), out.data_ptr(),
                                 last.data_ptr() if last is not None else None, B, T, D, code,
                                 _stream_ptr(stream), ctypes.byref(o) if o is not None else None)
    _check(rc, "lrscan_fwd")
    return out, last


def _check_host(shape, dtype, **tensors):
    for name, t in tensors.items():
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.is_cuda:
            raise ValueError(f"{name} must be a host (CPU) tensor; pin it for full copy speed")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if name == "last":
            if t.dtype != torch.float32 or tuple(t.shape) != (shape[0], shape[2]):
                raise ValueError("last must be fp32 [B, D]")
            continue
        if t.dtype != dtype or tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} must be {dtype} {tuple(shape)}")


def _host_like(t: torch.Tensor, shape=None, dtype=None) -> torch.Tensor:
    return torch.empty(shape if shape is not None else t.shape, dtype=dtype or t.dtype, pin_memory=True)


def lrscan_fwd_host(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None,
                    last: torch.Tensor | None = None, *, path=None, chunk_len=None, tile_variant=None):
    """Forward scan of host (CPU) tensors through the device (lrscan_fwd_host):
    copies in, kernels and copies out pipelined over batch-row chunks.  Outputs
    not given are allocated in page-locked memory.  Returns (out, last)."""
    if a.ndim != 3 or a.shape != b.shape:
        raise ValueError("lrscan expects matching [B, T, D] tensors")
    code = _dtype_code(a)
    B, T, D = a.shape
    out = _host_like(a) if out is None else out
    last = _host_like(a, (B, D), torch.float32) if last is None else last
    _check_host(a.shape, a.dtype, a=a, b=b, out=out, last=last)
    o = _opts(path, chunk_len, tile_variant, None)
    rc = lib().lrscan_fwd_host(a.data_ptr(), b.data_ptr(), out.data_ptr(), last.data_ptr(), B, T, D, code,
                               ctypes.byref(o) if o is not None else None)
    _check(rc, "lrscan_fwd_host")
    return out, last


def lrscan_bwd_host(a: torch.Tensor, out: torch.Tensor, grad_out: torch.Tensor,
                    grad_a: torch.Tensor | None = None, grad_b: torch.Tensor | None = None, *,
                    path=None, chunk_len=None, tile_variant=None):
    """Backward scan of host tensors through the device (lrscan_bwd_host);
    returns (grad_a, grad_b)."""
    if a.ndim != 3:
        raise ValueError("lrscan expects [B, T, D] tensors")
    code = _dtype_code(a)
    B, T, D = a.shape
    grad_a = _host_like(a) if grad_a is None else grad_a
    grad_b = _host_like(a) if grad_b is None else grad_b
    _check_host(a.shape, a.dtype, a=a, out=out, grad_out=grad_out, grad_a=grad_a, grad_b=grad_b)
    o = _opts(path, chunk_len, tile_variant, None)
    rc = lib().lrscan_bwd_host(a.data_ptr(), out.data_ptr(), grad_out.data_ptr(), grad_a.data_ptr(),
                               grad_b.data_ptr(), B, T, D, code, ctypes.byref(o) if o is not None else None)
    _check(rc, "lrscan_bwd_host")
    return grad_a, grad_b


def lrscan_fwd_bwd_host(a: torch.Tensor, b: torch.Tensor, grad_out: torch.Tensor, out=None, last=None,
                        grad_a=None, grad_b=None, *, path=None, chunk_len=None, tile_variant=None):
    """Forward then backward of host tensors through the device
    (lrscan_fwd_bwd_host; out stays on the device between them); returns
    (out, last, grad_a, grad_b)."""
    if a.ndim != 3 or a.shape != b.shape:
        raise ValueError("lrscan expects matching [B, T, D] tensors")
    code = _dtype_code(a)
    B, T, D = a.shape
    out = _host_like(a) if out is None else out
    last = _host_like(a, (B, D), torch.float32) if last is None else last
    grad_a = _host_like(a) if grad_a is None else grad_a
    grad_b = _host_like(a) if grad_b is None else grad_b
    _check_host(a.shape, a.dtype, a=a, b=b, grad_out=grad_out, out=out, last=last, grad_a=grad_a, grad_b=grad_b)
    o = _opts(path, chunk_len, tile_variant, None)
    rc = lib().lrscan_fwd_bwd_host(a.data_ptr(), b.data_ptr(), grad_out.data_ptr(), out.data_ptr(),
                                   last.data_ptr(), grad_a.data_ptr(), grad_b.data_ptr(), B, T, D, code,
                                   ctypes.byref(o) if o is not None else None)
    _check(rc, "lrscan_fwd_bwd_host")
    return out, last, grad_a, grad_b


def lrscan_bwd(a: torch.Tensor, out: torch.Tensor, grad_out: torch.Tensor,
               grad_a: torch.Tensor | None = None, grad_b: torch.Tensor | None = None, *,
               path=None, chunk_len=None, tile_variant=None, workspace=None, stream=None):
    """Reverse scan; returns (grad_a, grad_b) for the loss sum(grad_out * out)."""
    if a.ndim != 3:
        raise ValueError("lrscan expects [B, T, D] tensors")
    code = _dtype_code(a)
    B, T, D = a.shape
    if grad_a is None:
        grad_a = torch.empty_like(a)
    if grad_b is None:
        grad_b = torch.empty_like(a)
    _check_tensors(a.shape, a.dtype, a.device, a=a, out=out, grad_out=grad_out, grad_a=grad_a,
                   grad_b=grad_b)
    with torch.cuda.device(a.device):
        o = _opts(path, chunk_len, tile_variant, workspace)
        rc = lib().lrscan_bwd_ex(a.data_ptr(), out.data_ptr(), grad_out.data_ptr(), grad_a.data_ptr(),
                                 grad_b.data_ptr(), B, T, D, code, _stream_ptr(stream),
                                 ctypes.byref(o) if o is not None else None)
    _check(rc, "lrscan_bwd")
    return grad_a, grad_b


def _check_state_tensor(name, t, shape, dtype, device):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)}")
    return t.data_ptr()


def _state(a, h0=None, segment_pos=None, grad_last=None, grad_h0=None) -> State:
    B, T, D = a.shape
    st = State()
    st.h0 = _check_state_tensor("h0", h0, (B, D), torch.float32, a.device)
    st.segment_pos = _check_state_tensor("segment_pos", segment_pos, (B, T), torch.int32, a.device)
    st.grad_last = _check_state_tensor("grad_last", grad_last, (B, D), torch.float32, a.device)
    st.grad_h0 = _check_state_tensor("grad_h0", grad_h0, (B, D), torch.float32, a.device)
    return st


def lrscan_fwd_state(a: torch.Tensor, b: torch.Tensor, h0: torch.Tensor | None = None,
                     segment_pos: torch.Tensor | None = None, out: torch.Tensor | None = None,
                     last: torch.Tensor | None = None, *, path=None, chunk_len=None, tile_variant=None,
                     workspace=None, stream=None):
    """Forward scan from the fp32 [B, D] state h0, restarting where the int32
    [B, T] segment_pos is 0; returns (out, last)."""
    if a.ndim != 3 or a.shape != b.shape:
        raise ValueError("lrscan expects matching [B, T, D] tensors")
    code = _dtype_code(a)
    B, T, D = a.shape
    if out is None:
        out = torch.empty_like(b)
    if last is None:
        last = torch.empty((B, D), device=a.device, dtype=torch.float32)
    _check_tensors(a.shape, a.dtype, a.device, a=a, b=b, out=out, last=last)
    st = _state(a, h0=h0, segment_pos=segment_pos)
    with torch.cuda.device(a.device):
        o = _opts(path, chunk_len, tile_variant, workspace)
        rc = lib().lrscan_fwd_state(a.data_ptr(), b.data_ptr(), out.data_ptr(), last.data_ptr(),
                                    ctypes.byref(st), B, T, D, code, _stream_ptr(stream),
                                    ctypes.byref(o) if o is not None else None)
    _check(rc, "lrscan_fwd_state")
    return out, last


def lrscan_bwd_state(a: torch.Tensor, out: torch.Tensor, grad_out: torch.Tensor,
                     h0: torch.Tensor | None = None, segment_pos: torch.Tensor | None = None,
                     grad_last: torch.Tensor | None = None, grad_a: torch.Tensor | None = None,
                     grad_b: torch.Tensor | None = None, grad_h0: torch.Tensor | None = None, *,
                     want_grad_h0: bool = True, path=None, chunk_len=None, tile_variant=None, workspace=None,
                     stream=None):
    """Reverse scan of :func:`lrscan_fwd_state` for the loss
    sum(grad_out * out) + sum(grad_last * last); returns (grad_a, grad_b, grad_h0)
    (grad_h0 None when not wanted)."""
    if a.ndim != 3:
        raise ValueError("lrscan expects [B, T, D] tensors")
    code = _dtype_code(a)
    B, T, D = a.shape
    if grad_a is None:
        grad_a = torch.empty_like(a)
    if grad_b is None:
        grad_b = torch.empty_like(a)
    if grad_h0 is None and want_grad_h0:
        grad_h0 = torch.empty((B, D), device=a.device, dtype=torch.float32)
    _check_tensors(a.shape, a.dtype, a.device, a=a, out=out, grad_out=grad_out, grad_a=grad_a,
                   grad_b=grad_b)
    st = _state(a, h0=h0, segment_pos=segment_pos, grad_last=grad_last, grad_h0=grad_h0)
    with torch.cuda.device(a.device):
        o = _opts(path, chunk_len, tile_variant, workspace)
        rc = lib().lrscan_bwd_state(a.data_ptr(), out.data_ptr(), grad_out.data_ptr(), grad_a.data_ptr(),
                                    grad_b.data_ptr(), ctypes.byref(st), B, T, D, code, _stream_ptr(stream),
                                    ctypes.byref(o) if o is not None else None)
    _check(rc, "lrscan_bwd_state")
    return grad_a, grad_b, grad_h0


def lrscan_summary(a: torch.Tensor, x: torch.Tensor, segment_pos: torch.Tensor | None = None,
                   direction: str = "fwd", stream=None):
    """Per-lane affine map (P, Q), fp32 [B, D] each, of the whole sequence:
    h_{T-1} = P*h0 + Q (direction "fwd", x = b) or grad_h0 = P*grad_last + Q
    (direction "bwd", x = grad_out)."""
    if a.ndim != 3 or a.shape != x.shape:
        raise ValueError("lrscan expects matching [B, T, D] tensors")
    code = _dtype_code(a)
    B, T, D = a.shape
    _check_tensors(a.shape, a.dtype, a.device, a=a, x=x)
    seg = _check_state_tensor("segment_pos", segment_pos, (B, T), torch.int32, a.device)
    P = torch.empty((B, D), device=a.device, dtype=torch.float32)
    Q = torch.empty((B, D), device=a.device, dtype=torch.float32)
    with torch.cuda.device(a.device):
        rc = lib().lrscan_summary(a.data_ptr(), x.data_ptr(), P.data_ptr(), Q.data_ptr(), seg, B, T, D, code,
                                  {"fwd": 0, "bwd": 1}[direction], _stream_ptr(stream))
    _check(rc, "lrscan_summary")
    return P, Q


def lrscan_compose_maps(maps: torch.Tensor, rank: int, init: torch.Tensor | None = None,
                        direction: str = "fwd", stream=None) -> torch.Tensor:
    """Fold of the per-segment maps maps[r] = (P_r, Q_r) (fp32 [W, 2, B, D]) over
    init: segments 0..rank-1 ("fwd") or W-1..rank+1 ("bwd"); returns [B, D]."""
    if maps.ndim != 4 or maps.shape[1] != 2 or maps.dtype != torch.float32 or not maps.is_cuda:
        raise ValueError("maps must be a CUDA fp32 [W, 2, B, D] tensor")
    maps = maps.contiguous()
    W, _, B, D = maps.shape
    ip = _check_state_tensor("init", init, (B, D), torch.float32, maps.device)
    out = torch.empty((B, D), device=maps.device, dtype=torch.float32)
    with torch.cuda.device(maps.device):
        rc = lib().lrscan_compose_maps(maps.data_ptr(), W, rank, ip, out.data_ptr(), B, D,
                                       {"fwd": 0, "bwd": 1}[direction], _stream_ptr(stream))
    _check(rc, "lrscan_compose_maps")
    return out


def lrscan_cfwd(ar, ai, br, bi, *, out_r=None, out_i=None, last_r=None, last_i=None, want_last: bool = True,
                path=None, chunk_len=None, tile_variant=None, workspace=None, stream=None):
    """Complex forward scan on re/im planes [B, T, D]; returns
    (out_r, out_i, last_r, last_i) (last planes fp32 [B, D], or None)."""
    if ar.ndim != 3 or any(t.shape != ar.shape for t in (ai, br, bi)):
        raise ValueError("lrscan expects matching [B, T, D] planes")
    code = _dtype_code(ar)
    B, T, D = ar.shape
    out_r = torch.empty_like(ar) if out_r is None else out_r
    out_i = torch.empty_like(ar) if out_i is None else out_i
    if want_last:
        last_r = torch.empty((B, D), device=ar.device, dtype=torch.float32) if last_r is None else last_r
        last_i = torch.empty((B, D), device=ar.device, dtype=torch.float32) if last_i is None else last_i
    _check_tensors(ar.shape, ar.dtype, ar.device, ar=ar, ai=ai, br=br, bi=bi, out_r=out_r, out_i=out_i)
    for name, t in (("last_r", last_r), ("last_i", last_i)):
        if t is not None:
            _check_state_tensor(name, t, (B, D), torch.float32, ar.device)
    with torch.cuda.device(ar.device):
        o = _opts(path, chunk_len, tile_variant, workspace)
        rc = lib().lrscan_cfwd(ar.data_ptr(), ai.data_ptr(), br.data_ptr(), bi.data_ptr(), out_r.data_ptr(),
                               out_i.data_ptr(), last_r.data_ptr() if last_r is not None else None,
                               last_i.data_ptr() if last_i is not None else None, B, T, D, code,
                               _stream_ptr(stream), ctypes.byref(o) if o is not None else None)
    _check(rc, "lrscan_cfwd")
    return out_r, out_i, last_r, last_i


def lrscan_cbwd(ar, ai, out_r, out_i, grad_out_r, grad_out_i, *, grads=None, path=None, chunk_len=None,
                tile_variant=None, workspace=None, stream=None):
    """Complex reverse scan; returns (grad_ar, grad_ai, grad_br, grad_bi) for the
    loss sum(grad_out_r * out_r + grad_out_i * out_i)."""
    if ar.ndim != 3:
        raise ValueError("lrscan expects [B, T, D] planes")
    code = _dtype_code(ar)
    B, T, D = ar.shape
    grads = tuple(torch.empty_like(ar) for _ in range(4)) if grads is None else tuple(grads)
    _check_tensors(ar.shape, ar.dtype, ar.device, ar=ar, ai=ai, out_r=out_r, out_i=out_i, grad_out_r=grad_out_r,
                   grad_out_i=grad_out_i, grad_ar=grads[0], grad_ai=grads[1], grad_br=grads[2], grad_bi=grads[3])
    with torch.cuda.device(ar.device):
        o = _opts(path, chunk_len, tile_variant, workspace)
        rc = lib().lrscan_cbwd(ar.data_ptr(), ai.data_ptr(), out_r.data_ptr(), out_i.data_ptr(),
                               grad_out_r.data_ptr(), grad_out_i.data_ptr(), *[g.data_ptr() for g in grads],
                               B, T, D, code, _stream_ptr(stream), ctypes.byref(o) if o is not None else None)
    _check(rc, "lrscan_cbwd")
    return grads


def _cstate(ar, h0=None, segment_pos=None, grad_last=None, grad_h0=None) -> CState:
    B, T, D = ar.shape
    st = CState()
    pairs = (("h0", h0, ("h0_r", "h0_i")), ("grad_last", grad_last, ("grad_last_r", "grad_last_i")),
             ("grad_h0", grad_h0, ("grad_h0_r", "grad_h0_i")))
    for name, pair, fields in pairs:
        if pair is None:
            continue
        if len(pair) != 2:
            raise ValueError(f"{name} must be a (re, im) pair of tensors")
        for f, t in zip(fields, pair):
            setattr(st, f, _check_state_tensor(f, t, (B, D), torch.float32, ar.device))
    st.segment_pos = _check_state_tensor("segment_pos", segment_pos, (B, T), torch.int32, ar.device)
    return st


def lrscan_cfwd_state(ar, ai, br, bi, h0=None, segment_pos=None, *, out_r=None, out_i=None, last_r=None,
                      last_i=None, path=None, chunk_len=None, tile_variant=None, workspace=None, stream=None):
    """Complex forward scan from the fp32 (re, im) [B, D] state h0, restarting
    where the int32 [B, T] segment_pos is 0; returns (out_r, out_i, last_r,
    last_i).  Runs where the plan puts it: the tiled kernels, chunk
    streaming (few lanes, long sequences) or the chunked path."""
    if ar.ndim != 3 or any(t.shape != ar.shape for t in (ai, br, bi)):
        raise ValueError("lrscan expects matching [B, T, D] planes")
    code = _dtype_code(ar)
    B, T, D = ar.shape
    out_r = torch.empty_like(ar) if out_r is None else out_r
    out_i = torch.empty_like(ar) if out_i is None else out_i
    last_r = torch.empty((B, D), device=ar.device, dtype=torch.float32) if last_r is None else last_r
    last_i = torch.empty((B, D), device=ar.device, dtype=torch.float32) if last_i is None else last_i
    _check_tensors(ar.shape, ar.dtype, ar.device, ar=ar, ai=ai, br=br, bi=bi, out_r=out_r, out_i=out_i)
    for name, t in (("last_r", last_r), ("last_i", last_i)):
        _check_state_tensor(name, t, (B, D), torch.float32, ar.device)
    st = _cstate(ar, h0=h0, segment_pos=segment_pos)
    with torch.cuda.device(ar.device):
        o = _opts(path, chunk_len, tile_variant, workspace)
        rc = lib().lrscan_cfwd_state(ar.data_ptr(), ai.data_ptr(), br.data_ptr(), bi.data_ptr(), out_r.data_ptr(),
                                     out_i.data_ptr(), last_r.data_ptr(), last_i.data_ptr(), ctypes.byref(st),
                                     B, T, D, code, _stream_ptr(stream), ctypes.byref(o) if o is not None else None)
    _check(rc, "lrscan_cfwd_state")
    return out_r, out_i, last_r, last_i


def lrscan_cbwd_state(ar, ai, out_r, out_i, grad_out_r, grad_out_i, h0=None, segment_pos=None, grad_last=None, *,
                      grads=None, grad_h0=None, path=None, chunk_len=None, tile_variant=None, workspace=None,
                      stream=None):
    """Reverse scan of :func:`lrscan_cfwd_state` for the loss
    sum(Re(conj(grad_out) h)) + Re(conj(grad_last) last); returns
    (grad_ar, grad_ai, grad_br, grad_bi, grad_h0_r, grad_h0_i)."""
    if ar.ndim != 3:
        raise ValueError("lrscan expects [B, T, D] planes")
    code = _dtype_code(ar)
    B, T, D = ar.shape
    grads = tuple(torch.empty_like(ar) for _ in range(4)) if grads is None else tuple(grads)
    if grad_h0 is None:
        grad_h0 = tuple(torch.empty((B, D), device=ar.device, dtype=torch.float32) for _ in range(2))
    _check_tensors(ar.shape, ar.dtype, ar.device, ar=ar, ai=ai, out_r=out_r, out_i=out_i, grad_out_r=grad_out_r,
                   grad_out_i=grad_out_i, grad_ar=grads[0], grad_ai=grads[1], grad_br=grads[2], grad_bi=grads[3])
    st = _cstate(ar, h0=h0, segment_pos=segment_pos, grad_last=grad_last, grad_h0=grad_h0)
    with torch.cuda.device(ar.device):
        o = _opts(path, chunk_len, tile_variant, workspace)
        rc = lib().lrscan_cbwd_state(ar.data_ptr(), ai.data_ptr(), out_r.data_ptr(), out_i.data_ptr(),
                                     grad_out_r.data_ptr(), grad_out_i.data_ptr(), *[g.data_ptr() for g in grads],
                                     ctypes.byref(st), B, T, D, code, _stream_ptr(stream),
                                     ctypes.byref(o) if o is not None else None)
    _check(rc, "lrscan_cbwd_state")
    return (*grads, *grad_h0)


def lrscan_plan_complex(B: int, T: int, D: int, dtype="f32", direction: str = "fwd", aligned: bool = True,
                        path=None, tile_variant=None, chunk_len=None, state: bool = False) -> dict:
    """What the dispatcher would run for a complex scan (host only);
    state=True plans a call with carried state or resets
    (lrscan_plan_complex_state)."""
    code = {"f32": F32, "bf16": BF16}.get(dtype) if isinstance(dtype, str) else _DTYPES.get(dtype)
    if code is None:
        raise ValueError(f"unsupported dtype {dtype}")
    info = PlanInfo()
    o = _opts(path, chunk_len, tile_variant, None)
    fn = lib().lrscan_plan_complex_state if state else lib().lrscan_plan_complex
    rc = fn(B, T, D, code, 0 if direction == "fwd" else 1, int(aligned),
            ctypes.byref(o) if o is not None else None, ctypes.byref(info))
    _check(rc, "lrscan_plan_complex_state" if state else "lrscan_plan_complex")
    return info.as_dict()


def _gated_params(eta, nu_log, B, T, D, device):
    if not (isinstance(eta, torch.Tensor) and eta.is_cuda and eta.dtype == torch.float32
            and tuple(eta.shape) == (B, T) and eta.is_contiguous() and eta.device == device):
        raise ValueError(f"eta must be a contiguous CUDA fp32 tensor of shape {(B, T)}")
    if not (isinstance(nu_log, torch.Tensor) and nu_log.is_cuda and nu_log.dtype == torch.float32
            and tuple(nu_log.shape) == (D,) and nu_log.is_contiguous() and nu_log.device == device):
        raise ValueError(f"nu_log must be a contiguous CUDA fp32 tensor of shape {(D,)}")


def lrscan_fwd_gated(eta, nu_log, b, *, out=None, last=None, path=None, tile_variant=None, stream=None):
    """Scan with the decay generated as exp(-exp(nu_log[d]) * exp(eta[b, t]));
    eta fp32 [B, T], nu_log fp32 [D], b [B, T, D]; returns (out, last)."""
    if b.ndim != 3:
        raise ValueError("lrscan expects a [B, T, D] tensor b")
    code = _dtype_code(b)
    B, T, D = b.shape
    _gated_params(eta, nu_log, B, T, D, b.device)
    out = torch.empty_like(b) if out is None else out
    last = torch.empty((B, D), device=b.device, dtype=torch.float32) if last is None else last
    _check_tensors(b.shape, b.dtype, b.device, b=b, out=out, last=last)
    with torch.cuda.device(b.device):
        o = _opts(path, None, tile_variant, None)
        rc = lib().lrscan_fwd_gated(eta.data_ptr(), nu_log.data_ptr(), b.data_ptr(), out.data_ptr(), last.data_ptr(),
                                    B, T, D, code, _stream_ptr(stream), ctypes.byref(o) if o is not None else None)
    _check(rc, "lrscan_fwd_gated")
    return out, last


def lrscan_bwd_gated(eta, nu_log, out, grad_out, *, grad_b=None, path=None, tile_variant=None, workspace=None,
                     stream=None):
    """Reverse of :func:`lrscan_fwd_gated`; returns (grad_b, grad_eta, grad_nu_log)."""
    if out.ndim != 3:
        raise ValueError("lrscan expects [B, T, D] tensors")
    code = _dtype_code(out)
    B, T, D = out.shape
    _gated_params(eta, nu_log, B, T, D, out.device)
    grad_b = torch.empty_like(out) if grad_b is None else grad_b
    _check_tensors(out.shape, out.dtype, out.device, out=out, grad_out=grad_out, grad_b=grad_b)
    grad_eta = torch.empty((B, T), device=out.device, dtype=torch.float32)
    grad_nu = torch.empty((D,), device=out.device, dtype=torch.float32)
    with torch.cuda.device(out.device):
        o = _opts(path, None, tile_variant, workspace)
        rc = lib().lrscan_bwd_gated(eta.data_ptr(), nu_log.data_ptr(), out.data_ptr(), grad_out.data_ptr(),
                                    grad_b.data_ptr(), grad_eta.data_ptr(), grad_nu.data_ptr(), B, T, D, code,
                                    _stream_ptr(stream), ctypes.byref(o) if o is not None else None)
    _check(rc, "lrscan_bwd_gated")
    return grad_b, grad_eta, grad_nu


def lrscan_plan_gated(B: int, T: int, D: int, dtype="f32", direction: str = "fwd", aligned: bool = True,
                      path=None, tile_variant=None) -> dict:
    code = {"f32": F32, "bf16": BF16}.get(dtype) if isinstance(dtype, str) else _DTYPES.get(dtype)
    if code is None:
        raise ValueError(f"unsupported dtype {dtype}")
    info = PlanInfo()
    o = _opts(path, None, tile_variant, None)
    rc = lib().lrscan_plan_gated(B, T, D, code, 0 if direction == "fwd" else 1, int(aligned),
                                 ctypes.byref(o) if o is not None else None, ctypes.byref(info))
    _check(rc, "lrscan_plan_gated")
    return info.as_dict()


def lrscan_gated_workspace_bytes(B: int, T: int, D: int) -> int:
    return lib().lrscan_gated_workspace_bytes(B, T, D)


def lrscan_plan(B: int, T: int, D: int, dtype: torch.dtype | str = torch.float32, direction: str = "fwd",
                aligned: bool = True, path=None, chunk_len=None, tile_variant=None, state: bool = False) -> dict:
    """What the dispatcher would run for this call (host only; no launch);
    state=True plans a call with carried state or resets (lrscan_plan_state)."""
    code = {"f32": F32, "bf16": BF16}.get(dtype) if isinstance(dtype, str) else _DTYPES.get(dtype)
    if code is None:
        raise ValueError(f"unsupported dtype {dtype}")
    info = PlanInfo()
    o = _opts(path, chunk_len, tile_variant, None)
    fn = lib().lrscan_plan_state if state else lib().lrscan_plan
    rc = fn(B, T, D, code, 0 if direction == "fwd" else 1, int(aligned),
            ctypes.byref(o) if o is not None else None, ctypes.byref(info))
    _check(rc, "lrscan_plan_state" if state else "lrscan_plan")
    return info.as_dict()


def lrscan_num_variants(path: str, dtype: str = "f32", direction: str = "fwd") -> int:
    return lib().lrscan_num_variants(PATHS[path], {"f32": F32, "bf16": BF16}[dtype],
                                     0 if direction == "fwd" else 1)


def lrscan_workspace_bytes(B: int, T: int, D: int, chunk_len: int = 64) -> int:
    return lib().lrscan_workspace_bytes(B, T, D, chunk_len)


def lrscan_sync_check(stream=None) -> int:
    """Synchronize the stream and return (and clear) any device-side error code."""
    lib().lrscan_set_stream(_stream_ptr(stream))
    return lib().lrscan_sync_check()


def lrscan_set_wait_timeout_ns(ns: int) -> None:
    _check(lib().lrscan_set_wait_timeout_ns(ns), "lrscan_set_wait_timeout_ns")


def lrscan_selftest_wait_timeout(timeout_ns: int, stream=None) -> int:
    lib().lrscan_set_stream(_stream_ptr(stream))
    return lib().lrscan_selftest_wait_timeout(timeout_ns)


class LinearRecurrenceScan(torch.autograd.Function):
    """Autograd wrapper: out = scan(a, b); backward through lrscan_bwd."""

    @staticmethod
    def forward(ctx, a, b, path=None, chunk_len=None):
        a, b = a.contiguous(), b.contiguous()
        out, _ = lrscan_fwd(a, b, want_last=False, path=path, chunk_len=chunk_len)
        ctx.save_for_backward(a, out)
        ctx.opts = (path, chunk_len)
        return out

    @staticmethod
    def backward(ctx, grad_out):
        a, out = ctx.saved_tensors
        path, chunk_len = ctx.opts
        ga, gb = lrscan_bwd(a, out, grad_out.contiguous(), path=path, chunk_len=chunk_len)
        return ga, gb, None, None


def scan(a: torch.Tensor, b: torch.Tensor, path=None, chunk_len=None) -> torch.Tensor:
    """Differentiable h_t = a_t*h_{t-1} + b_t over [B, T, D] (fp32 or bf16 storage)."""
    return LinearRecurrenceScan.apply(a, b, path, chunk_len)


class LinearRecurrenceScanState(torch.autograd.Function):
    """Autograd wrapper of the state-carrying scan: (out, last) = scan(a, b, h0,
    segment_pos); gradients flow to a, b and h0 from both outputs."""

    @staticmethod
    def forward(ctx, a, b, h0, segment_pos, path=None, chunk_len=None):
        a, b = a.contiguous(), b.contiguous()
        h0c = h0.contiguous() if h0 is not None else None
        seg = segment_pos.contiguous() if segment_pos is not None else None
        out, last = lrscan_fwd_state(a, b, h0=h0c, segment_pos=seg, path=path, chunk_len=chunk_len)
        ctx.save_for_backward(a, out, h0c, seg)
        ctx.opts = (path, chunk_len)
        ctx.mark_non_differentiable(*(() if seg is None else (seg,)))
        return out, last

    @staticmethod
    def backward(ctx, grad_out, grad_last):
        a, out, h0, seg = ctx.saved_tensors
        path, chunk_len = ctx.opts
        if grad_out is None:
            grad_out = torch.zeros_like(out)
        ga, gb, gh0 = lrscan_bwd_state(a, out, grad_out.contiguous(), h0=h0, segment_pos=seg,
                                       grad_last=grad_last.contiguous() if grad_last is not None else None,
                                       path=path, chunk_len=chunk_len)
        return ga, gb, (gh0 if h0 is not None else None), None, None, None


def scan_state(a: torch.Tensor, b: torch.Tensor, h0: torch.Tensor | None = None,
               segment_pos: torch.Tensor | None = None, path=None, chunk_len=None):
    """Differentiable state-carrying scan; returns (out, last) with last fp32 [B, D]."""
    return LinearRecurrenceScanState.apply(a, b, h0, segment_pos, path, chunk_len)


class ComplexScan(torch.autograd.Function):
    """Autograd wrapper of the complex scan: (out_r, out_i) = scan(ar, ai, br, bi)."""

    @staticmethod
    def forward(ctx, ar, ai, br, bi, path=None):
        ar, ai, br, bi = (t.contiguous() for t in (ar, ai, br, bi))
        out_r, out_i, _, _ = lrscan_cfwd(ar, ai, br, bi, want_last=False, path=path)
        ctx.save_for_backward(ar, ai, out_r, out_i)
        ctx.path = path
        return out_r, out_i

    @staticmethod
    def backward(ctx, grad_out_r, grad_out_i):
        ar, ai, out_r, out_i = ctx.saved_tensors
        gr = torch.zeros_like(out_r) if grad_out_r is None else grad_out_r.contiguous()
        gi = torch.zeros_like(out_i) if grad_out_i is None else grad_out_i.contiguous()
        return (*lrscan_cbwd(ar, ai, out_r, out_i, gr, gi, path=ctx.path), None)


def complex_scan(ar, ai, br, bi, path=None):
    """Differentiable complex diagonal scan on re/im planes; returns (out_r, out_i)."""
    return ComplexScan.apply(ar, ai, br, bi, path)


class ComplexScanState(torch.autograd.Function):
    """Autograd wrapper of the state-carrying complex scan: (out_r, out_i,
    last_r, last_i) = scan(ar, ai, br, bi, h0 = (h0_r, h0_i), segment_pos);
    gradients flow to the decays, the inputs and h0 from every output."""

    @staticmethod
    def forward(ctx, ar, ai, br, bi, h0_r, h0_i, segment_pos, chunk_len=None):
        ar, ai, br, bi = (t.contiguous() for t in (ar, ai, br, bi))
        B, _, D = ar.shape
        if (h0_r is None) != (h0_i is None):
            zero = torch.zeros((B, D), device=ar.device, dtype=torch.float32)
            h0_r = zero if h0_r is None else h0_r
            h0_i = zero if h0_i is None else h0_i
        h0 = None if h0_r is None else (h0_r.contiguous(), h0_i.contiguous())
        seg = segment_pos.contiguous() if segment_pos is not None else None
        out_r, out_i, last_r, last_i = lrscan_cfwd_state(ar, ai, br, bi, h0=h0, segment_pos=seg, chunk_len=chunk_len)
        ctx.save_for_backward(ar, ai, out_r, out_i, *(h0 if h0 is not None else (None, None)), seg)
        ctx.chunk_len = chunk_len
        ctx.has_h0 = h0 is not None
        ctx.mark_non_differentiable(*(() if seg is None else (seg,)))
        return out_r, out_i, last_r, last_i

    @staticmethod
    def backward(ctx, g_out_r, g_out_i, g_last_r, g_last_i):
        ar, ai, out_r, out_i, h0_r, h0_i, seg = ctx.saved_tensors
        gr = torch.zeros_like(out_r) if g_out_r is None else g_out_r.contiguous()
        gi = torch.zeros_like(out_i) if g_out_i is None else g_out_i.contiguous()
        gl = None
        if g_last_r is not None or g_last_i is not None:
            z = torch.zeros((ar.shape[0], ar.shape[2]), device=ar.device, dtype=torch.float32)
            gl = ((z if g_last_r is None else g_last_r).contiguous(), (z if g_last_i is None else g_last_i).contiguous())
        h0 = (h0_r, h0_i) if ctx.has_h0 else None
        g = lrscan_cbwd_state(ar, ai, out_r, out_i, gr, gi, h0=h0, segment_pos=seg, grad_last=gl,
                              chunk_len=ctx.chunk_len)
        gh0 = (g[4], g[5]) if ctx.has_h0 else (None, None)
        return (*g[:4], *gh0, None, None)


def complex_scan_state(ar, ai, br, bi, h0=None, segment_pos=None, chunk_len=None):
    """Differentiable state-carrying complex scan; h0 is an fp32 (re, im) pair
    of [B, D] tensors or None; returns (out_r, out_i, last_r, last_i)."""
    h0_r, h0_i = (None, None) if h0 is None else h0
    return ComplexScanState.apply(ar, ai, br, bi, h0_r, h0_i, segment_pos, chunk_len)


class GatedScan(torch.autograd.Function):
    """Autograd wrapper of the generated-decay scan: out = scan(eta, nu_log, b)."""

    @staticmethod
    def forward(ctx, eta, nu_log, b, path=None):
        eta, nu_log, b = eta.contiguous(), nu_log.contiguous(), b.contiguous()
        out, _ = lrscan_fwd_gated(eta, nu_log, b, path=path)
        ctx.save_for_backward(eta, nu_log, out)
        ctx.path = path
        return out

    @staticmethod
    def backward(ctx, grad_out):
        eta, nu_log, out = ctx.saved_tensors
        gb, geta, gnu = lrscan_bwd_gated(eta, nu_log, out, grad_out.contiguous(), path=ctx.path)
        return geta, gnu, gb, None


def gated_scan(eta, nu_log, b, path=None):
    """Differentiable scan whose decays exp(-exp(nu_log[d]) * exp(eta[b, t])) are
    generated in the kernel; returns out [B, T, D]."""
    return GatedScan.apply(eta, nu_log, b, path)
