"""Python binding of librd, the GB300 (sm_103a) ragged_dot library.

Argument marshalling only: every step of the path runs in the CUDA kernels
of ``librd.so`` behind the C ABI declared in ``include/rd.h``.  torch is used
for device memory and the current stream, nothing else.  There is no CPU or
library fallback: if the library is missing, every call raises.

Functions (same names as the C ABI, without the ``rd_`` prefix):

* ``ragged_dot(lhs, rhs, group_sizes, ...)``             -> out [m, n] (or [m, n/2] with GLU)
* ``ragged_dot_trans_rhs(lhs, rhs, group_sizes, ...)``   -> out [m, k]
* ``ragged_dot_trans_rhs_glu_bwd(d_out, rhs, fused, group_sizes, ...)`` -> [d_gate | d_up] [m, 2f]
* ``trans_ragged_dot(x, y, group_sizes, ...)``           -> out [g_local, k, n]
* ``trans_ragged_dot_f32(x, y, group_sizes, ..., accumulate=False)`` -> f32 out [g_local, k, n]
* ``dw_workspace_bytes(device)``                         -> the dw calls' workspace size
* ``trans_ragged_dot_no_alloc(x, y, group_sizes, ...)``  -> dw with no allocation (library scratch)
* ``glu_fwd(fused, limit=None)``                         -> out [rows, f]
* ``glu_bwd(fused, d_out, limit=None)``                  -> d_fused [rows, 2f]
* ``unsort_bwd_rows(g, y, w, limit=None)``                -> (grad [rows, hidden], dot [rows])
* ``set_tuning(...)``, ``get_tuning()``, ``tuning(...)``  -> the process-wide launch overrides
* ``status_bits(status)``, ``check_status(status)``       -> read a status word (names, or raise)

Every tensor of a call must sit on one CUDA device; the call runs on that
device's current stream (or ``stream``).  A ``status`` word (a one-element
int32 CUDA tensor) collects the device-side status bits; without one a call
whose bounded waits ran out cannot be told from a completed one.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = [
    "load", "lib_path", "ragged_dot", "ragged_dot_trans_rhs", "ragged_dot_trans_rhs_glu_bwd",
    "trans_ragged_dot", "trans_ragged_dot_f32", "trans_ragged_dot_no_alloc", "dw_workspace_bytes",
    "glu_fwd", "glu_bwd", "unsort_bwd_rows", "RdError", "EPI_NONE", "EPI_SILU_GLU",
    "STATUS_NEG_SIZE", "STATUS_OVERFLOW", "STATUS_TIMEOUT", "MAX_GROUPS",
    "VARIANT_AUTO", "VARIANT_SINGLE", "VARIANT_PAIR", "set_tuning", "get_tuning", "tuning",
    "status_bits", "check_status",
]

EPI_NONE = 0
EPI_SILU_GLU = 1
STATUS_NEG_SIZE = 1
STATUS_OVERFLOW = 2
STATUS_TIMEOUT = 4
MAX_GROUPS = 1024
VARIANT_AUTO = 0
VARIANT_SINGLE = 1
VARIANT_PAIR = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "librd.so")
_lib = None


class _Tuning(ctypes.Structure):
    _fields_ = [("gemm_variant", ctypes.c_int32), ("band_rows", ctypes.c_int32),
                ("wait_timeout_ns", ctypes.c_uint64), ("reserved", ctypes.c_int32 * 2)]


class RdError(RuntimeError):
    """A non-OK rd_status returned by the library."""

    def __init__(self, code: int, message: str):
        super().__init__(message)
        self.code = code


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load librd.so (built by ``expert_ffn_ragged_gb300.build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"librd.so is not built ({_LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i64, i32, ip = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    grouped = [vp, vp, vp, i64, i64, i64, ip, i32, i32, i32, ip]
    lib.rd_ragged_dot.argtypes = grouped + [ctypes.c_int, ip, vp]
    lib.rd_ragged_dot_trans_rhs.argtypes = grouped + [ip, vp]
    lib.rd_ragged_dot_trans_rhs_glu_bwd.argtypes = [vp] + grouped + [ip, vp]
    sz = ctypes.c_size_t
    lib.rd_trans_ragged_dot.argtypes = grouped + [vp, sz, ip, vp]
    lib.rd_trans_ragged_dot_f32.argtypes = grouped + [i32, vp, sz, ip, vp]
    lib.rd_trans_ragged_dot_no_alloc.argtypes = grouped + [ip, vp]
    lib.rd_trans_ragged_dot_no_alloc.restype = ctypes.c_int
    lib.rd_trans_ragged_dot_workspace_size.argtypes = [ctypes.c_void_p]
    lib.rd_trans_ragged_dot_workspace_size.restype = ctypes.c_int
    lib.rd_glu_fwd.argtypes = [vp, vp, i64, i64, ip, vp]
    lib.rd_glu_bwd.argtypes = [vp, vp, vp, i64, i64, ip, vp]
    lib.rd_unsort_bwd_rows.argtypes = [vp, vp, vp, vp, vp, i64, i64, ip, vp]
    for fn in (lib.rd_ragged_dot, lib.rd_ragged_dot_trans_rhs,
               lib.rd_ragged_dot_trans_rhs_glu_bwd, lib.rd_trans_ragged_dot,
               lib.rd_trans_ragged_dot_f32,
               lib.rd_glu_fwd, lib.rd_glu_bwd, lib.rd_unsort_bwd_rows):
        fn.restype = ctypes.c_int
    lib.rd_set_tuning.argtypes = [ctypes.c_void_p]
    lib.rd_get_tuning.argtypes = [ctypes.c_void_p]
    lib.rd_set_tuning.restype = ctypes.c_int
    lib.rd_get_tuning.restype = ctypes.c_int
    lib.rd_status_string.argtypes = [ctypes.c_int]
    lib.rd_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(code: int, what: str):
    if code != 0:
        msg = _lib.rd_status_string(code).decode()
        raise RdError(code, f"{what}: {msg}")


_STATUS_NAMES = ((STATUS_NEG_SIZE, "STATUS_NEG_SIZE: a group size < 0 was treated as 0"),
                 (STATUS_OVERFLOW, "STATUS_OVERFLOW: the group sizes add up past m; boundaries clamped"),
                 (STATUS_TIMEOUT, "STATUS_TIMEOUT: a bounded wait in a kernel ran out; outputs incomplete"))


def status_bits(status) -> list:
    """The names of the bits set in a status word (waits for the work queued before)."""
    v = int(status.item())
    return [name for bit, name in _STATUS_NAMES if v & bit]


def check_status(status, allow=STATUS_NEG_SIZE | STATUS_OVERFLOW):
    """Raise RdError if the status word holds a bit outside ``allow`` (by default only
    STATUS_TIMEOUT raises: the size bits report data the kernels clamped and handled).
    Reading the word waits for the calls that report into it."""
    v = int(status.item())
    bad = v & ~allow
    if bad:
        names = [name for bit, name in _STATUS_NAMES if bad & bit]
        raise RdError(-1, "; ".join(names) or f"status bits {bad:#x}")
    return v


_torch_module = None


def _torch():
    """torch, imported once (a call's host work is part of its latency)."""
    global _torch_module
    if _torch_module is None:
        import torch

        _torch_module = torch
    return _torch_module


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


_raw_stream = None


def _stream(stream, device):
    """The raw cudaStream_t of ``stream`` (default: the device's current stream)."""
    global _raw_stream
    torch = _torch()
    if stream is None:
        if _raw_stream is None:
            # the current stream's handle without building a Stream object (the
            # public route costs ~2 us a call); fall back to it where absent
            _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", False)
        if _raw_stream:
            return _raw_stream(device.index if device.index is not None
                               else torch.cuda.current_device())
        stream = torch.cuda.current_stream(device)
    elif stream.device != device:
        raise ValueError("stream is on another device than the tensors")
    return stream.cuda_stream


class _on_device:
    """Make ``device`` current for the call (the library launches on the current device)."""

    __slots__ = ("idx", "prev")

    def __init__(self, device):
        self.idx = device.index if device.index is not None else _torch().cuda.current_device()
        self.prev = None

    def __enter__(self):
        torch = _torch()
        cur = torch.cuda.current_device()
        if cur != self.idx:
            self.prev = cur
            torch.cuda.set_device(self.idx)

    def __exit__(self, *exc):
        if self.prev is not None:
            _torch().cuda.set_device(self.prev)


def _same_device(device, *tensors):
    idx = device.index if device.index is not None else _torch().cuda.current_device()
    for t in tensors:
        if t is not None and t.get_device() != idx:
            raise ValueError(f"all tensors of a call must be on {device} (one is on {t.device})")


def _bf16_2d(t, name):
    torch = _torch()

    if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D bf16 CUDA tensor")


def _bf16_3d(t, name, what):
    torch = _torch()

    if t.dtype != torch.bfloat16 or t.dim() != 3 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {what} bf16 CUDA tensor")


def _out(t, shape, dtype, name="out"):
    """A caller-supplied output must match exactly: the library only sees its pointer."""
    if (tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_cuda
            or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous {list(shape)} {dtype} CUDA tensor")


def _scalar_i32(t, name):
    torch = _torch()

    if t is not None and (t.dtype != torch.int32 or t.numel() != 1 or not t.is_cuda):
        raise ValueError(f"{name} must be a one-element int32 CUDA tensor")


def _group_args(group_sizes, limit, status):
    torch = _torch()

    if (group_sizes.dtype != torch.int32 or group_sizes.dim() != 1 or not group_sizes.is_cuda
            or not group_sizes.is_contiguous()):
        raise ValueError("group_sizes must be a contiguous 1-D int32 CUDA tensor")
    _scalar_i32(limit, "limit")
    _scalar_i32(status, "status")


def _fused_width(fused):
    rows, w = fused.shape
    if w % 2:
        raise ValueError("fused must have an even width: [rows, 2f] = [gate | up]")
    return rows, w // 2


def set_tuning(variant: Optional[int] = None, band_rows: Optional[int] = None,
               wait_timeout_ns: Optional[int] = None):
    """Set the process-wide launch overrides of rd_set_tuning; None leaves a field as it is.

    variant: VARIANT_AUTO / VARIANT_SINGLE / VARIANT_PAIR; band_rows: rows per
    band of the forward / dx tile order (0 = default); wait_timeout_ns: bound
    of each wait inside the kernels (0 = default).  A CUDA graph keeps the
    values in force when it was captured.
    """
    lib = load()
    cur = _Tuning()
    _check(lib.rd_get_tuning(ctypes.byref(cur)), "rd_get_tuning")
    if variant is not None:
        cur.gemm_variant = int(variant)
    if band_rows is not None:
        cur.band_rows = int(band_rows)
    if wait_timeout_ns is not None:
        cur.wait_timeout_ns = int(wait_timeout_ns)
    _check(lib.rd_set_tuning(ctypes.byref(cur)), "rd_set_tuning")


def get_tuning() -> dict:
    lib = load()
    cur = _Tuning()
    _check(lib.rd_get_tuning(ctypes.byref(cur)), "rd_get_tuning")
    return {"variant": cur.gemm_variant, "band_rows": cur.band_rows,
            "wait_timeout_ns": cur.wait_timeout_ns}


class tuning:
    """Context manager: the overrides of ``set_tuning`` inside, the previous values after."""

    def __init__(self, **kw):
        self.kw = kw
        self.saved = None

    def __enter__(self):
        self.saved = get_tuning()
        set_tuning(**self.kw)
        return self

    def __exit__(self, *exc):
        s = self.saved
        set_tuning(s["variant"], s["band_rows"], s["wait_timeout_ns"])


def ragged_dot(lhs, rhs, group_sizes, group_offset: int = 0, limit=None, epilogue: int = EPI_NONE,
               out=None, status=None, stream=None):
    """Grouped forward out[i] = lhs[i] @ rhs[group(i) - group_offset] (see rd_ragged_dot)."""
    torch = _torch()

    lib = load()
    _bf16_2d(lhs, "lhs")
    _group_args(group_sizes, limit, status)
    _bf16_3d(rhs, "rhs", "[g_local, k, n]")
    m, k = lhs.shape
    g_local, k2, n = rhs.shape
    if k2 != k:
        raise ValueError("lhs and rhs disagree on k")
    n_out = n // 2 if epilogue == EPI_SILU_GLU else n
    dev = lhs.device
    if out is None:
        out = torch.empty((m, n_out), dtype=torch.bfloat16, device=dev)
    _out(out, (m, n_out), torch.bfloat16)
    _same_device(dev, rhs, out, group_sizes, limit, status)
    with _on_device(dev):
        code = lib.rd_ragged_dot(_ptr(lhs), _ptr(rhs), _ptr(out), m, k, n, _ptr(group_sizes),
                                 group_sizes.numel(), group_offset, g_local, _ptr(limit),
                                 int(epilogue), _ptr(status), _stream(stream, dev))
    _check(code, "rd_ragged_dot")
    return out


def ragged_dot_trans_rhs(lhs, rhs, group_sizes, group_offset: int = 0, limit=None, out=None,
                         status=None, stream=None):
    """out[i] = lhs[i] @ rhs[group(i) - group_offset]^T; lhs [m, n], rhs [g_local, k, n]."""
    torch = _torch()

    lib = load()
    _bf16_2d(lhs, "lhs")
    _group_args(group_sizes, limit, status)
    _bf16_3d(rhs, "rhs", "[g_local, k, n]")
    m, n = lhs.shape
    g_local, k, n2 = rhs.shape
    if n2 != n:
        raise ValueError("lhs and rhs disagree on n")
    dev = lhs.device
    if out is None:
        out = torch.empty((m, k), dtype=torch.bfloat16, device=dev)
    _out(out, (m, k), torch.bfloat16)
    _same_device(dev, rhs, out, group_sizes, limit, status)
    with _on_device(dev):
        code = lib.rd_ragged_dot_trans_rhs(_ptr(lhs), _ptr(rhs), _ptr(out), m, k, n,
                                           _ptr(group_sizes), group_sizes.numel(), group_offset,
                                           g_local, _ptr(limit), _ptr(status), _stream(stream, dev))
    _check(code, "rd_ragged_dot_trans_rhs")
    return out


def ragged_dot_trans_rhs_glu_bwd(d_out, rhs, fused, group_sizes, group_offset: int = 0, limit=None,
                                 out=None, status=None, stream=None):
    """[d_gate | d_up] of an expert FFN from its output gradient, through the down projection.

    d_out [m, n], rhs [g_local, f, n] (down weights), fused [m, 2f] (saved gate | up).
    """
    torch = _torch()

    lib = load()
    _bf16_2d(d_out, "d_out")
    _bf16_2d(fused, "fused")
    _group_args(group_sizes, limit, status)
    _bf16_3d(rhs, "rhs", "[g_local, f, n]")
    m, n = d_out.shape
    g_local, f, n2 = rhs.shape
    if n2 != n or fused.shape != (m, 2 * f):
        raise ValueError("shapes disagree: d_out [m, n], rhs [g, f, n], fused [m, 2f]")
    dev = d_out.device
    if out is None:
        out = torch.empty((m, 2 * f), dtype=torch.bfloat16, device=dev)
    _out(out, (m, 2 * f), torch.bfloat16)
    _same_device(dev, rhs, fused, out, group_sizes, limit, status)
    with _on_device(dev):
        code = lib.rd_ragged_dot_trans_rhs_glu_bwd(
            _ptr(d_out), _ptr(rhs), _ptr(fused), _ptr(out), m, f, n, _ptr(group_sizes),
            group_sizes.numel(), group_offset, g_local, _ptr(limit), _ptr(status),
            _stream(stream, dev))
    _check(code, "rd_ragged_dot_trans_rhs_glu_bwd")
    return out


_ws_bytes = {}


def dw_workspace_bytes(device=None) -> int:
    """Bytes of the dw workspace (rd_trans_ragged_dot_workspace_size) on a CUDA device."""
    torch = _torch()

    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if dev.index not in _ws_bytes:
        lib = load()
        n = ctypes.c_size_t(0)
        with _on_device(dev):
            _check(lib.rd_trans_ragged_dot_workspace_size(ctypes.byref(n)),
                   "rd_trans_ragged_dot_workspace_size")
        _ws_bytes[dev.index] = n.value
    return _ws_bytes[dev.index]


def _dw_workspace(workspace, dev, stream):
    """The workspace argument of the dw calls: "auto" allocates one for this call."""
    torch = _torch()

    if workspace is None:
        return None
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError('workspace must be "auto", None or a uint8 CUDA tensor')
        ws = torch.empty(dw_workspace_bytes(dev), dtype=torch.uint8, device=dev)
        if stream is not None and stream != torch.cuda.current_stream(dev):
            ws.record_stream(stream)     # freed after the call: keep it until the stream is done
        return ws
    if workspace.dtype != torch.uint8 or not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 CUDA tensor")
    return workspace


def _dw_args(x, y, group_sizes, group_offset, g_local, limit, status):
    _bf16_2d(x, "x")
    _bf16_2d(y, "y")
    _group_args(group_sizes, limit, status)
    m, k = x.shape
    m2, n = y.shape
    if m2 != m:
        raise ValueError("x and y disagree on m")
    if g_local is None:
        g_local = group_sizes.numel() - group_offset
    return m, k, n, g_local


def trans_ragged_dot(x, y, group_sizes, group_offset: int = 0, g_local: Optional[int] = None,
                     limit=None, out=None, status=None, stream=None, workspace="auto"):
    """out[j] = x[rows_j]^T @ y[rows_j] for the local groups; x [m, k], y [m, n].

    workspace: "auto" (a workspace of dw_workspace_bytes() allocated for the
    call), None (the form without one), or a caller's uint8 CUDA tensor.
    """
    torch = _torch()

    lib = load()
    m, k, n, g_local = _dw_args(x, y, group_sizes, group_offset, g_local, limit, status)
    dev = x.device
    if out is None:
        out = torch.empty((g_local, k, n), dtype=torch.bfloat16, device=dev)
    _out(out, (g_local, k, n), torch.bfloat16)
    ws = _dw_workspace(workspace, dev, stream)
    _same_device(dev, y, out, group_sizes, limit, status, ws)
    with _on_device(dev):
        code = lib.rd_trans_ragged_dot(_ptr(x), _ptr(y), _ptr(out), m, k, n, _ptr(group_sizes),
                                       group_sizes.numel(), group_offset, g_local, _ptr(limit),
                                       _ptr(ws), 0 if ws is None else ws.numel(), _ptr(status),
                                       _stream(stream, dev))
    _check(code, "rd_trans_ragged_dot")
    return out


def trans_ragged_dot_no_alloc(x, y, group_sizes, group_offset: int = 0,
                              g_local: Optional[int] = None, limit=None, out=None, status=None,
                              stream=None):
    """trans_ragged_dot for callers that cannot allocate device memory at the call.

    The same per-group-descriptor dw as trans_ragged_dot with a workspace, its
    scratch taken from an array inside the library (see
    rd_trans_ragged_dot_no_alloc: up to 256 SMs; calls that overlap on the GPU
    race on the array; make the first call on a device outside stream capture).
    Pass ``out`` to allocate nothing at all.
    """
    torch = _torch()

    lib = load()
    m, k, n, g_local = _dw_args(x, y, group_sizes, group_offset, g_local, limit, status)
    dev = x.device
    if out is None:
        out = torch.empty((g_local, k, n), dtype=torch.bfloat16, device=dev)
    _out(out, (g_local, k, n), torch.bfloat16)
    _same_device(dev, y, out, group_sizes, limit, status)
    with _on_device(dev):
        code = lib.rd_trans_ragged_dot_no_alloc(_ptr(x), _ptr(y), _ptr(out), m, k, n,
                                                _ptr(group_sizes), group_sizes.numel(),
                                                group_offset, g_local, _ptr(limit), _ptr(status),
                                                _stream(stream, dev))
    _check(code, "rd_trans_ragged_dot_no_alloc")
    return out


def trans_ragged_dot_f32(x, y, group_sizes, group_offset: int = 0, g_local: Optional[int] = None,
                         limit=None, out=None, accumulate: bool = False, status=None, stream=None,
                         workspace="auto"):
    """out[j] (+)= x[rows_j]^T @ y[rows_j] in f32; ``accumulate`` adds into ``out``.

    An accumulating call whose status reports STATUS_TIMEOUT has added some
    tiles and not others: its output is unusable (a retry would add twice).
    """
    torch = _torch()

    lib = load()
    m, k, n, g_local = _dw_args(x, y, group_sizes, group_offset, g_local, limit, status)
    dev = x.device
    if out is None:
        if accumulate:
            raise ValueError("accumulate needs an existing out buffer")
        out = torch.empty((g_local, k, n), dtype=torch.float32, device=dev)
    _out(out, (g_local, k, n), torch.float32)
    ws = _dw_workspace(workspace, dev, stream)
    _same_device(dev, y, out, group_sizes, limit, status, ws)
    with _on_device(dev):
        code = lib.rd_trans_ragged_dot_f32(_ptr(x), _ptr(y), _ptr(out), m, k, n,
                                           _ptr(group_sizes), group_sizes.numel(), group_offset,
                                           g_local, _ptr(limit), 1 if accumulate else 0,
                                           _ptr(ws), 0 if ws is None else ws.numel(),
                                           _ptr(status), _stream(stream, dev))
    _check(code, "rd_trans_ragged_dot_f32")
    return out


def glu_fwd(fused, limit=None, out=None, stream=None):
    """silu(gate) * up over the rows below limit of a fused [rows, 2f] buffer."""
    torch = _torch()

    lib = load()
    _bf16_2d(fused, "fused")
    _scalar_i32(limit, "limit")
    rows, f = _fused_width(fused)
    dev = fused.device
    if out is None:
        out = torch.empty((rows, f), dtype=torch.bfloat16, device=dev)
    _out(out, (rows, f), torch.bfloat16)
    _same_device(dev, out, limit)
    with _on_device(dev):
        code = lib.rd_glu_fwd(_ptr(fused), _ptr(out), rows, f, _ptr(limit), _stream(stream, dev))
    _check(code, "rd_glu_fwd")
    return out


def glu_bwd(fused, d_out, limit=None, out=None, stream=None):
    """[d_gate | d_up] for the rows below limit; fused [rows, 2f], d_out [rows, f]."""
    torch = _torch()

    lib = load()
    _bf16_2d(fused, "fused")
    _bf16_2d(d_out, "d_out")
    rows, f = _fused_width(fused)
    if d_out.shape != (rows, f):
        raise ValueError("d_out must be [rows, f]")
    _scalar_i32(limit, "limit")
    dev = fused.device
    if out is None:
        out = torch.empty((rows, 2 * f), dtype=torch.bfloat16, device=dev)
    _out(out, (rows, 2 * f), torch.bfloat16)
    _same_device(dev, d_out, out, limit)
    with _on_device(dev):
        code = lib.rd_glu_bwd(_ptr(fused), _ptr(d_out), _ptr(out), rows, f, _ptr(limit),
                              _stream(stream, dev))
    _check(code, "rd_glu_bwd")
    return out


def unsort_bwd_rows(g, y, w, limit=None, grad=None, dot=None, stream=None):
    """Weighted gradient bf16(f32(g) * w) and f32 row dot sum(g * y) over rows below limit."""
    torch = _torch()

    lib = load()
    _bf16_2d(g, "g")
    _bf16_2d(y, "y")
    rows, hidden = g.shape
    if y.shape != g.shape:
        raise ValueError("g and y must have the same shape")
    if (w.dtype != torch.float32 or tuple(w.shape) != (rows,) or not w.is_cuda
            or not w.is_contiguous()):
        raise ValueError("w must be a contiguous [rows] float32 CUDA tensor")
    _scalar_i32(limit, "limit")
    dev = g.device
    if grad is None:
        grad = torch.empty_like(g)
    if dot is None:
        dot = torch.empty((rows,), dtype=torch.float32, device=dev)
    _out(grad, (rows, hidden), torch.bfloat16, "grad")
    _out(dot, (rows,), torch.float32, "dot")
    _same_device(dev, y, w, grad, dot, limit)
    with _on_device(dev):
        code = lib.rd_unsort_bwd_rows(_ptr(g), _ptr(y), _ptr(w), _ptr(grad), _ptr(dot), rows,
                                      hidden, _ptr(limit), _stream(stream, dev))
    _check(code, "rd_unsort_bwd_rows")
    return grad, dot
