"""ctypes binding of libscan (include/libscan.h).

Argument marshalling only: every function checks shapes and dtypes of torch
CUDA tensors, allocates the outputs with torch, passes raw device pointers and
the current stream to the C entry point of the same name, and raises
``ScanError`` on a non-zero status. All arithmetic runs in libscan's kernels.
There is no fallback: if libscan.so is missing or no GPU is present, the call
fails.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libscan.so")

SCAN_OK = 0
SCAN_ERR_INVALID_ARG = 1
SCAN_ERR_UNSUPPORTED = 2
SCAN_ERR_ALIGNMENT = 3
SCAN_ERR_WORKSPACE = 4
SCAN_ERR_CUDA = 5
SCAN_ERR_TIMEOUT = 6
SCAN_ERR_SEQLENS = 7

SCAN_F32 = 0
SCAN_BF16 = 1

SCAN_VARIANT_AUTO = 0
SCAN_VARIANT_STATIONARY = 1
SCAN_VARIANT_LOOKBACK = 2
SCAN_VARIANT_STREAM = 3

SCAN_OP_FWD = 0
SCAN_OP_BWD = 1
SCAN_OP_BIDIR_FWD = 2
SCAN_OP_BIDIR_BWD = 3
SCAN_OP_LOG_FWD = 4
SCAN_OP_AFFINE_FWD = 5
SCAN_OP_AFFINE_BWD = 6
SCAN_OP_LOG_BWD = 7

SCAN_COPY_VEC = 0
SCAN_COPY_TMA = 1

EXPORTED = (
    "scan_status_string", "scan_version", "scan_workspace_bytes", "scan_workspace_init",
    "scan_get_device_status", "scan_fwd", "scan_bwd", "scan_bidir_fwd", "scan_bidir_bwd",
    "scan_log_fwd", "scan_log_bwd", "affine_scan_fwd", "affine_scan_bwd", "affine_prefix_fwd",
    "affine_prefix_bwd", "gdn_checkpoint_bytes", "gdn_fwd", "gdn_workspace_bytes", "gdn_bwd",
    "scan_fwd_noalloc", "scan_noalloc_device_status", "scan_step_host", "scan_copy",
    "rglru_fwd", "rglru_bwd",
)


class ScanError(RuntimeError):
    """A libscan entry point returned a non-zero scan_status."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class ScanOpts(ctypes.Structure):
    _fields_ = [
        ("variant", ctypes.c_int32),
        ("chunk", ctypes.c_int32),
        ("rows_per_cta", ctypes.c_int32),
        ("test_stall", ctypes.c_int32),
        ("wait_limit_s", ctypes.c_double),
        ("cu_seqlens_host", ctypes.POINTER(ctypes.c_int32)),
        ("segments", ctypes.c_int32),
        ("stages", ctypes.c_int32),
    ]


class HostIO(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("a", "x", "h0", "dh", "h", "da", "dx", "dh0")]


class DeviceIO(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("a", "x", "h0", "dh", "h", "da", "dx", "dh0")]


_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t
_opt = ctypes.POINTER(ScanOpts)

_SIGS = {
    "scan_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "scan_version": ([], ctypes.c_int32),
    "scan_workspace_bytes": ([ctypes.c_int, _i64, _i64, _i64, _i32, _i32, _opt], _sz),
    "scan_workspace_init": ([_vp, _sz, _vp], ctypes.c_int),
    "scan_get_device_status": ([_vp, _vp], ctypes.c_int),
    "scan_fwd": ([_vp, _vp, _vp, _vp, _i32, _vp, _i64, _i64, _i64, ctypes.c_int, _i32, _opt,
                  _vp, _sz, _vp], ctypes.c_int),
    "scan_bwd": ([_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_int,
                  _i32, _opt, _vp, _sz, _vp], ctypes.c_int),
    "scan_bidir_fwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _i64, _i64, _i64,
                        ctypes.c_int, _opt, _vp, _sz, _vp], ctypes.c_int),
    "scan_bidir_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp,
                        _vp, _vp, _i64, _i64, _i64, ctypes.c_int, _opt, _vp, _sz, _vp],
                       ctypes.c_int),
    "scan_log_fwd": ([_vp, _vp, _vp, _vp, _i32, _vp, _i64, _i64, _i64, _i32, _opt, _vp, _sz,
                      _vp], ctypes.c_int),
    "scan_log_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _i64, _i64, _i64, _i32,
                      _opt, _vp, _sz, _vp], ctypes.c_int),
    "affine_scan_fwd": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _opt, _vp, _sz, _vp],
                        ctypes.c_int),
    "affine_scan_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _opt,
                         _vp, _sz, _vp], ctypes.c_int),
    "affine_prefix_fwd": ([_vp, _vp, _i64, _i64, _i64, _i32, _opt, _vp, _sz, _vp], ctypes.c_int),
    "gdn_checkpoint_bytes": ([_i64, _i64, _i64, _i64, _i64], ctypes.c_size_t),
    "gdn_fwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _vp, _sz,
                 _vp], ctypes.c_int),
    "gdn_workspace_bytes": ([_i64, _i64, _i64, _i64, _i64], ctypes.c_size_t),
    "scan_step_host": ([ctypes.POINTER(HostIO), ctypes.POINTER(DeviceIO), _i64, _i64, _i64,
                        ctypes.c_int, _i32, _opt, _vp, _sz, _vp], ctypes.c_int),
    "gdn_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                 _i64, _vp, _sz, _vp], ctypes.c_int),
    "affine_prefix_bwd": ([_vp, _vp, _vp, _vp, _i32, _i64, _i64, _i64, _i32, _opt, _vp, _sz, _vp],
                          ctypes.c_int),
    "scan_fwd_noalloc": ([_vp, _vp, _vp, _vp, _i32, _vp, _i64, _i64, _i64, ctypes.c_int, _i32,
                          _vp], ctypes.c_int),
    "scan_noalloc_device_status": ([_vp], ctypes.c_int),
    "rglru_fwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_int, _vp],
                  ctypes.c_int),
    "rglru_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                   _i64, ctypes.c_int, _vp], ctypes.c_int),
    "scan_copy": ([_vp, _vp, _sz, _i32, _vp, _vp], ctypes.c_int),
}

_lock = threading.Lock()
_lib_handle = None


def lib() -> ctypes.CDLL:
    """The loaded libscan.so (raises if it has not been built)."""
    global _lib_handle
    if _lib_handle is None:
        with _lock:
            if _lib_handle is None:
                if not os.path.exists(LIB_PATH):
                    raise ImportError(
                        f"{LIB_PATH} is missing: build it with "
                        "`python -c 'import __graft_entry__ as g; g.build()'`")
                h = ctypes.CDLL(LIB_PATH)
                for name, (args, res) in _SIGS.items():
                    fn = getattr(h, name)
                    fn.argtypes = args
                    fn.restype = res
                _lib_handle = h
    return _lib_handle


def status_string(status: int) -> str:
    return lib().scan_status_string(int(status)).decode()


def _call(device, name: str, *args):
    """Call entry point `name` with `device` current: the library launches on
    the current device, which must be the one holding the tensors."""
    with torch.cuda.device(device):
        return getattr(lib(), name)(*args)


def _check(status: int, where: str) -> None:
    if status != SCAN_OK:
        raise ScanError(status, where)


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _opts(opts) -> Optional[ScanOpts]:
    if opts is None:
        return None
    if isinstance(opts, ScanOpts):
        return opts
    o = ScanOpts()
    known = {name for name, _ in ScanOpts._fields_}
    for k, v in dict(opts).items():
        if k not in known:  # a ctypes structure would keep a misspelt name as a plain attribute
            raise ValueError(f"unknown scan option {k!r}; options are {sorted(known)}")
        if k == "cu_seqlens_host":
            arr = (ctypes.c_int32 * len(v))(*[int(e) for e in v])
            o._keep = arr  # keep the host copy alive for the call
            o.cu_seqlens_host = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))
        else:
            setattr(o, k, v)
    return o


def _optref(o: Optional[ScanOpts]):
    return None if o is None else ctypes.byref(o)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SCAN_F32
    if t.dtype == torch.bfloat16:
        return SCAN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: fp32 or bf16 expected")


def _need(t: Optional[torch.Tensor], name: str, *, dtype=None, shape=None, device=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _scalar_dims(a: torch.Tensor, cu_seqlens):
    if cu_seqlens is None:
        if a.dim() != 3:
            raise ValueError("dense scan expects [B, C, T]")
        return a.shape[0], a.shape[1], a.shape[2], 0
    if a.dim() != 2:
        raise ValueError("packed scan expects [C, T] with cu_seqlens")
    _need(cu_seqlens, "cu_seqlens", dtype=torch.int32, device=a.device)
    return 1, a.shape[0], a.shape[1], cu_seqlens.numel() - 1


class _Workspaces:
    """One zeroed workspace per (device, stream), grown on demand."""

    def __init__(self):
        self._buf = {}
        self._lk = threading.Lock()

    def get(self, nbytes: int, device: torch.device, stream: ctypes.c_void_p) -> torch.Tensor:
        key = (device.index, stream.value)
        with self._lk:
            buf = self._buf.get(key)
            if buf is None or buf.numel() < nbytes:
                size = max(nbytes, 4096)
                # The caching allocator orders a block's reuse by torch's current
                # stream only, while the library uses the buffer on `stream`:
                # wait for the device before a smaller buffer is given back (a
                # kernel on `stream` may still read it) and before a new block,
                # which may still be in use by work queued on another stream,
                # is zeroed on `stream`. Buffers only grow, so this is rare.
                torch.cuda.synchronize(device)
                buf = torch.empty(size, dtype=torch.uint8, device=device)
                _check(_call(device, "scan_workspace_init", _ptr(buf), size, stream),
                       "scan_workspace_init")
                self._buf[key] = buf
            return buf

    def current(self, device, stream):
        return self._buf.get((device.index, stream.value))


_ws = _Workspaces()


def workspace_for(op: int, B: int, C: int, T: int, k: int, v: int, opts, device, stream):
    o = _opts(opts)
    n = lib().scan_workspace_bytes(op, B, C, T, k, v, _optref(o))
    # 0 means the call itself will reject its arguments; give it a header-sized
    # workspace so that it reports its own, more precise status
    n = max(int(n), 4096)
    return _ws.get(n, device, stream), n, o


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def scan_version() -> int:
    return int(lib().scan_version())


def scan_status_string(status: int) -> str:
    return status_string(status)


def scan_workspace_bytes(op: int, B: int, C: int, T: int, k: int = 0, v: int = 0, opts=None) -> int:
    return int(lib().scan_workspace_bytes(op, B, C, T, k, v, _optref(_opts(opts))))


def scan_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    """Zero a caller-owned workspace (a CUDA uint8 tensor) on `stream`."""
    _need(workspace, "workspace")
    _check(_call(workspace.device, "scan_workspace_init", _ptr(workspace),
                 workspace.numel() * workspace.element_size(), _stream(stream, workspace.device)),
           "scan_workspace_init")


def scan_get_device_status(device=None, stream=None) -> int:
    """Sticky device status of the workspace used on (device, stream); resets it."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    s = _stream(stream, device)
    buf = _ws.current(device, s)
    if buf is None:
        return SCAN_OK
    return int(_call(device, "scan_get_device_status", _ptr(buf), s))


def scan_fwd(a, x, h0=None, cu_seqlens=None, reverse=False, *, out=None, opts=None, stream=None):
    """h_t = a_t h_{t-1} + x_t (reverse: h_t = a_t h_{t+1} + x_t). Returns h (fp32)."""
    _need(a, "a")
    dev = a.device
    dt = _dtype_code(a)
    B, C, T, n = _scalar_dims(a, cu_seqlens)
    _need(x, "x", dtype=a.dtype, shape=a.shape, device=dev)
    _need(h0, "h0", dtype=torch.float32, shape=(n, C) if cu_seqlens is not None else (B, C),
          device=dev)
    h = out if out is not None else torch.empty(a.shape, dtype=torch.float32, device=dev)
    _need(h, "out", dtype=torch.float32, shape=a.shape, device=dev)
    s = _stream(stream, dev)
    ws, nb, o = workspace_for(SCAN_OP_FWD, B, C, T, 0, 0, opts, dev, s)
    st = _call(dev, "scan_fwd", _ptr(a), _ptr(x), _ptr(h0), _ptr(cu_seqlens), n, _ptr(h), B, C, T, dt,
                        int(bool(reverse)), _optref(o), _ptr(ws), ws.numel(), s)
    _check(st, "scan_fwd")
    return h


def scan_bwd(a, h, dh, h0=None, cu_seqlens=None, reverse=False, *, out=None, opts=None,
             stream=None, need_dh0=True):
    """Backward of L = sum dh * h. Returns (da, dx, dh0) with da, dx in a's dtype."""
    _need(a, "a")
    dev = a.device
    dt = _dtype_code(a)
    B, C, T, n = _scalar_dims(a, cu_seqlens)
    _need(h, "h", dtype=torch.float32, shape=a.shape, device=dev)
    _need(dh, "dh", dtype=torch.float32, shape=a.shape, device=dev)
    h0_shape = (n, C) if cu_seqlens is not None else (B, C)
    _need(h0, "h0", dtype=torch.float32, shape=h0_shape, device=dev)
    if out is not None:
        da, dx, dh0 = out
    else:
        da = torch.empty_like(a)
        dx = torch.empty_like(a)
        dh0 = torch.empty(h0_shape, dtype=torch.float32, device=dev) if need_dh0 else None
    _need(da, "da", dtype=a.dtype, shape=a.shape, device=dev)
    _need(dx, "dx", dtype=a.dtype, shape=a.shape, device=dev)
    _need(dh0, "dh0", dtype=torch.float32, shape=h0_shape, device=dev)
    s = _stream(stream, dev)
    ws, nb, o = workspace_for(SCAN_OP_BWD, B, C, T, 0, 0, opts, dev, s)
    st = _call(dev, "scan_bwd", _ptr(a), _ptr(h), _ptr(dh), _ptr(h0), _ptr(cu_seqlens), n, _ptr(da),
                        _ptr(dx), _ptr(dh0), B, C, T, dt, int(bool(reverse)), _optref(o),
                        _ptr(ws), ws.numel(), s)
    _check(st, "scan_bwd")
    return da, dx, dh0


def scan_step_host(a, x, dh, h0=None, *, out, device, pieces=0, opts=None, stream=None):
    """scan_fwd then scan_bwd on dense rows held in host memory, pipelined over
    row pieces (copies overlap the scans). a, x, dh, h0: host tensors (pinned
    for overlap); out = (h, da, dx, dh0) host tensors for the results (dh0 None
    when h0 is None); device = (a, x, h0, dh, h, da, dx, dh0) device buffers of
    the same shapes on the device that runs the step. Returns out."""
    if a.dim() != 3:
        raise ValueError("scan_step_host takes dense [B, C, T] rows")
    B, C, T = a.shape
    dt = _dtype_code(a)
    h, da, dx, dh0 = out
    d_a, d_x, d_h0, d_dh, d_h, d_da, d_dx, d_dh0 = device
    for name, t in (("a", a), ("x", x), ("dh", dh), ("h", h), ("da", da), ("dx", dx)):
        if t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (B, C, T):
            raise ValueError(f"scan_step_host: host tensor {name} must be contiguous [B, C, T]")
    for name, t in (("h0", h0), ("dh0", dh0)):
        if t is not None and (t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (B, C)):
            raise ValueError(f"scan_step_host: host tensor {name} must be contiguous [B, C]")
    dev = d_a.device
    for name, t, like in (("a", d_a, a), ("x", d_x, x), ("dh", d_dh, dh), ("h", d_h, h),
                          ("da", d_da, da), ("dx", d_dx, dx), ("h0", d_h0, h0),
                          ("dh0", d_dh0, dh0)):
        if like is None:
            continue
        _need(t, "device " + name, dtype=like.dtype, shape=like.shape, device=dev)
    if x.dtype != a.dtype or da.dtype != a.dtype or dx.dtype != a.dtype:
        raise ValueError("scan_step_host: a, x, da, dx share one dtype")
    p = lambda t: None if t is None else t.data_ptr()
    hio = HostIO(p(a), p(x), p(h0), p(dh), p(h), p(da), p(dx), p(dh0))
    dio = DeviceIO(p(d_a), p(d_x), p(d_h0) if h0 is not None else None, p(d_dh), p(d_h), p(d_da),
                   p(d_dx), p(d_dh0) if dh0 is not None else None)
    s = _stream(stream, dev)
    np_ = pieces if pieces else min(8, B * C)
    rows = -(-(B * C) // max(np_, 1))
    o = ScanOpts()  # a copy: the caller's options are not modified
    src = _opts(opts)
    if src is not None:
        ctypes.memmove(ctypes.byref(o), ctypes.byref(src), ctypes.sizeof(ScanOpts))
    if o.variant == SCAN_VARIANT_AUTO:
        o.variant = SCAN_VARIANT_STATIONARY
    ws, nb, _ = workspace_for(SCAN_OP_BWD, 1, rows, T, 0, 0, o, dev, s)
    st = _call(dev, "scan_step_host", ctypes.byref(hio), ctypes.byref(dio), B, C, T, dt, int(pieces),
                              _optref(o), _ptr(ws), ws.numel(), s)
    _check(st, "scan_step_host")
    return out


def scan_bidir_fwd(af, xf, ar, xr, h0f=None, h0r=None, cu_seqlens=None, *, out=None, opts=None,
                   stream=None):
    """Causal branch over (af, xf) and reverse branch over (ar, xr). Returns (hf, hr)."""
    _need(af, "af")
    dev = af.device
    dt = _dtype_code(af)
    B, C, T, n = _scalar_dims(af, cu_seqlens)
    for t, nm in ((xf, "xf"), (ar, "ar"), (xr, "xr")):
        _need(t, nm, dtype=af.dtype, shape=af.shape, device=dev)
    h0_shape = (n, C) if cu_seqlens is not None else (B, C)
    _need(h0f, "h0f", dtype=torch.float32, shape=h0_shape, device=dev)
    _need(h0r, "h0r", dtype=torch.float32, shape=h0_shape, device=dev)
    if out is not None:
        hf, hr = out
    else:
        hf = torch.empty(af.shape, dtype=torch.float32, device=dev)
        hr = torch.empty(af.shape, dtype=torch.float32, device=dev)
    _need(hf, "hf", dtype=torch.float32, shape=af.shape, device=dev)
    _need(hr, "hr", dtype=torch.float32, shape=af.shape, device=dev)
    s = _stream(stream, dev)
    ws, nb, o = workspace_for(SCAN_OP_BIDIR_FWD, B, C, T, 0, 0, opts, dev, s)
    st = _call(dev, "scan_bidir_fwd", _ptr(af), _ptr(xf), _ptr(ar), _ptr(xr), _ptr(h0f), _ptr(h0r),
                              _ptr(cu_seqlens), n, _ptr(hf), _ptr(hr), B, C, T, dt, _optref(o),
                              _ptr(ws), ws.numel(), s)
    _check(st, "scan_bidir_fwd")
    return hf, hr


def scan_bidir_bwd(af, hf, dhf, ar, hr, dhr, h0f=None, h0r=None, cu_seqlens=None, *, out=None,
                   opts=None, stream=None):
    """Backward of both branches. Returns (daf, dxf, dh0f, dar, dxr, dh0r)."""
    _need(af, "af")
    dev = af.device
    dt = _dtype_code(af)
    B, C, T, n = _scalar_dims(af, cu_seqlens)
    _need(ar, "ar", dtype=af.dtype, shape=af.shape, device=dev)
    for t, nm in ((hf, "hf"), (dhf, "dhf"), (hr, "hr"), (dhr, "dhr")):
        _need(t, nm, dtype=torch.float32, shape=af.shape, device=dev)
    h0_shape = (n, C) if cu_seqlens is not None else (B, C)
    _need(h0f, "h0f", dtype=torch.float32, shape=h0_shape, device=dev)
    _need(h0r, "h0r", dtype=torch.float32, shape=h0_shape, device=dev)
    if out is not None:
        daf, dxf, dh0f, dar, dxr, dh0r = out
    else:
        daf, dxf, dar, dxr = (torch.empty_like(af) for _ in range(4))
        dh0f = torch.empty(h0_shape, dtype=torch.float32, device=dev)
        dh0r = torch.empty(h0_shape, dtype=torch.float32, device=dev)
    s = _stream(stream, dev)
    ws, nb, o = workspace_for(SCAN_OP_BIDIR_BWD, B, C, T, 0, 0, opts, dev, s)
    st = _call(dev, "scan_bidir_bwd", _ptr(af), _ptr(hf), _ptr(dhf), _ptr(h0f), _ptr(ar), _ptr(hr),
                              _ptr(dhr), _ptr(h0r), _ptr(cu_seqlens), n, _ptr(daf), _ptr(dxf),
                              _ptr(dh0f), _ptr(dar), _ptr(dxr), _ptr(dh0r), B, C, T, dt,
                              _optref(o), _ptr(ws), ws.numel(), s)
    _check(st, "scan_bidir_bwd")
    return daf, dxf, dh0f, dar, dxr, dh0r


def scan_log_fwd(log_a, log_x, log_h0=None, cu_seqlens=None, reverse=False, *, out=None, opts=None,
                 stream=None):
    """h_t = exp(l_t), l_t = log(exp(l_{t-1} + log_a_t) + exp(log_x_t)). Returns h (fp32)."""
    _need(log_a, "log_a", dtype=torch.float32)
    dev = log_a.device
    B, C, T, n = _scalar_dims(log_a, cu_seqlens)
    _need(log_x, "log_x", dtype=torch.float32, shape=log_a.shape, device=dev)
    _need(log_h0, "log_h0", dtype=torch.float32,
          shape=(n, C) if cu_seqlens is not None else (B, C), device=dev)
    h = out if out is not None else torch.empty(log_a.shape, dtype=torch.float32, device=dev)
    _need(h, "out", dtype=torch.float32, shape=log_a.shape, device=dev)
    s = _stream(stream, dev)
    ws, nb, o = workspace_for(SCAN_OP_LOG_FWD, B, C, T, 0, 0, opts, dev, s)
    st = _call(dev, "scan_log_fwd", _ptr(log_a), _ptr(log_x), _ptr(log_h0), _ptr(cu_seqlens), n, _ptr(h),
                            B, C, T, int(bool(reverse)), _optref(o), _ptr(ws), ws.numel(), s)
    _check(st, "scan_log_fwd")
    return h


def scan_log_bwd(log_a, log_x, h, dh, log_h0=None, cu_seqlens=None, reverse=False, *, out=None,
                 opts=None, stream=None, need_dh0=True):
    """Backward of L = sum dh * h for h = scan_log_fwd(log_a, log_x, log_h0, ...).

    Returns (dlog_a, dlog_x, dlog_h0), all fp32."""
    _need(log_a, "log_a", dtype=torch.float32)
    dev = log_a.device
    B, C, T, n = _scalar_dims(log_a, cu_seqlens)
    for t, name in ((log_x, "log_x"), (h, "h"), (dh, "dh")):
        _need(t, name, dtype=torch.float32, shape=log_a.shape, device=dev)
    h0_shape = (n, C) if cu_seqlens is not None else (B, C)
    _need(log_h0, "log_h0", dtype=torch.float32, shape=h0_shape, device=dev)
    if out is not None:
        dla, dlx, dlh0 = out
    else:
        dla = torch.empty_like(log_a)
        dlx = torch.empty_like(log_a)
        dlh0 = torch.empty(h0_shape, dtype=torch.float32, device=dev) if need_dh0 else None
    _need(dla, "dlog_a", dtype=torch.float32, shape=log_a.shape, device=dev)
    _need(dlx, "dlog_x", dtype=torch.float32, shape=log_a.shape, device=dev)
    _need(dlh0, "dlog_h0", dtype=torch.float32, shape=h0_shape, device=dev)
    s = _stream(stream, dev)
    ws, nb, o = workspace_for(SCAN_OP_LOG_BWD, B, C, T, 0, 0, opts, dev, s)
    st = _call(dev, "scan_log_bwd", _ptr(log_a), _ptr(log_x), _ptr(h), _ptr(dh), _ptr(log_h0),
                            _ptr(cu_seqlens), n, _ptr(dla), _ptr(dlx), _ptr(dlh0), B, C, T,
                            int(bool(reverse)), _optref(o), _ptr(ws), ws.numel(), s)
    _check(st, "scan_log_bwd")
    return dla, dlx, dlh0


def _affine_dims(A, Bm):
    if A.dim() != 5 or Bm.dim() != 5:
        raise ValueError("affine scan expects A [B,T,N,k,k] and Bm [B,T,N,k,v]")
    B, T, N, k, k2 = A.shape
    if k2 != k or tuple(Bm.shape[:4]) != (B, T, N, k):
        raise ValueError("affine scan: A [B,T,N,k,k] and Bm [B,T,N,k,v] disagree")
    return B, T, N, k, Bm.shape[4]


def affine_scan_fwd(A, Bm, h0=None, *, out=None, opts=None, stream=None):
    """H_t = A_t H_{t-1} + B_t. Returns H [B,T,N,k,v] (fp32)."""
    _need(A, "A", dtype=torch.float32)
    dev = A.device
    _need(Bm, "Bm", dtype=torch.float32, device=dev)
    B, T, N, k, v = _affine_dims(A, Bm)
    _need(h0, "h0", dtype=torch.float32, shape=(B, N, k, v), device=dev)
    H = out if out is not None else torch.empty(Bm.shape, dtype=torch.float32, device=dev)
    _need(H, "out", dtype=torch.float32, shape=Bm.shape, device=dev)
    s = _stream(stream, dev)
    ws, nb, o = workspace_for(SCAN_OP_AFFINE_FWD, B, N, T, k, v, opts, dev, s)
    st = _call(dev, "affine_scan_fwd", _ptr(A), _ptr(Bm), _ptr(h0), _ptr(H), B, T, N, k, v, _optref(o),
                               _ptr(ws), ws.numel(), s)
    _check(st, "affine_scan_fwd")
    return H


def affine_scan_bwd(A, H, dH, h0=None, *, out=None, opts=None, stream=None):
    """Backward of L = sum <dH_t, H_t>. Returns (dA, dB, dh0)."""
    _need(A, "A", dtype=torch.float32)
    dev = A.device
    _need(H, "H", dtype=torch.float32, device=dev)
    B, T, N, k, v = _affine_dims(A, H)
    _need(dH, "dH", dtype=torch.float32, shape=H.shape, device=dev)
    _need(h0, "h0", dtype=torch.float32, shape=(B, N, k, v), device=dev)
    if out is not None:
        dA, dB, dh0 = out
    else:
        dA = torch.empty_like(A)
        dB = torch.empty_like(H)
        dh0 = torch.empty((B, N, k, v), dtype=torch.float32, device=dev)
    s = _stream(stream, dev)
    ws, nb, o = workspace_for(SCAN_OP_AFFINE_BWD, B, N, T, k, v, opts, dev, s)
    st = _call(dev, "affine_scan_bwd", _ptr(A), _ptr(H), _ptr(dH), _ptr(h0), _ptr(dA), _ptr(dB),
                               _ptr(dh0), B, T, N, k, v, _optref(o), _ptr(ws), ws.numel(), s)
    _check(st, "affine_scan_bwd")
    return dA, dB, dh0


def affine_prefix_fwd(A, *, out=None, opts=None, stream=None):
    """Abar_t = A_t A_{t-1} ... A_0 per lane. Returns Abar [B,T,N,k,k] (fp32)."""
    _need(A, "A", dtype=torch.float32)
    if A.dim() != 5 or A.shape[3] != A.shape[4]:
        raise ValueError("affine_prefix_fwd expects A [B,T,N,k,k]")
    dev = A.device
    B, T, N, k, _ = A.shape
    Abar = out if out is not None else torch.empty_like(A)
    _need(Abar, "out", dtype=torch.float32, shape=A.shape, device=dev)
    s = _stream(stream, dev)
    ws, nb, o = workspace_for(SCAN_OP_AFFINE_FWD, B, N, T, k, k, opts, dev, s)
    st = _call(dev, "affine_prefix_fwd", _ptr(A), _ptr(Abar), B, T, N, k, _optref(o), _ptr(ws),
                                 ws.numel(), s)
    _check(st, "affine_prefix_fwd")
    return Abar


def affine_prefix_bwd(A, Abar, dAbar, dA=None, *, accumulate=False, opts=None, stream=None):
    """Backward of L = sum <dAbar_t, Abar_t>: returns dA, written (or, with
    accumulate=True, added into the given dA)."""
    _need(A, "A", dtype=torch.float32)
    dev = A.device
    for t, name in ((Abar, "Abar"), (dAbar, "dAbar")):
        _need(t, name, dtype=torch.float32, shape=A.shape, device=dev)
    if dA is None:
        if accumulate:
            raise ValueError("accumulate=True needs the dA to add into")
        dA = torch.empty_like(A)
    _need(dA, "dA", dtype=torch.float32, shape=A.shape, device=dev)
    B, T, N, k, _ = A.shape
    s = _stream(stream, dev)
    ws, nb, o = workspace_for(SCAN_OP_AFFINE_BWD, B, N, T, k, k, opts, dev, s)
    st = _call(dev, "affine_prefix_bwd", _ptr(A), _ptr(Abar), _ptr(dAbar), _ptr(dA), int(bool(accumulate)),
                                 B, T, N, k, _optref(o), _ptr(ws), ws.numel(), s)
    _check(st, "affine_prefix_bwd")
    return dA


def gdn_checkpoint_bytes(B, H, T, S, D) -> int:
    return int(lib().gdn_checkpoint_bytes(B, H, T, S, D))


def _gdn_dims(alpha, b, v, c):
    _need(alpha, "alpha", dtype=torch.float32)
    if alpha.dim() != 3 or b.dim() != 4 or v.dim() != 4:
        raise ValueError("gdn expects alpha [B,H,T], b, c [B,H,T,S], v [B,H,T,D]")
    B, H, T = alpha.shape
    S, D = b.shape[-1], v.shape[-1]
    dev = alpha.device
    _need(b, "b", dtype=torch.float32, shape=(B, H, T, S), device=dev)
    _need(c, "c", dtype=torch.float32, shape=(B, H, T, S), device=dev)
    _need(v, "v", dtype=torch.float32, shape=(B, H, T, D), device=dev)
    return B, H, T, S, D


def gdn_fwd(alpha, b, v, c, h0=None, *, checkpoints=True, out=None, workspace=None,
            stream=None):
    """o_t = h_t^T c_t with h_t = alpha_t h_{t-1} + b_t v_t^T. Returns (o, ckpt),
    ckpt being the backward's checkpoint buffer: allocated (checkpoints=True),
    the given fp32 tensor of gdn_checkpoint_bytes() bytes, or None (False).
    workspace: a device tensor of at least gdn_workspace_bytes() bytes
    (allocated here when None)."""
    B, H, T, S, D = _gdn_dims(alpha, b, v, c)
    dev = alpha.device
    _need(h0, "h0", dtype=torch.float32, shape=(B, H, S, D), device=dev)
    o = out if out is not None else torch.empty((B, H, T, D), dtype=torch.float32, device=dev)
    _need(o, "out", dtype=torch.float32, shape=(B, H, T, D), device=dev)
    ckpt = None
    n = gdn_checkpoint_bytes(B, H, T, S, D) // 4
    if isinstance(checkpoints, torch.Tensor):
        ckpt = checkpoints
        _need(ckpt, "checkpoints", dtype=torch.float32, device=dev)
        if ckpt.numel() < n or not ckpt.is_contiguous():
            raise ValueError(f"checkpoints: needs {n} contiguous floats")
    elif checkpoints:
        ckpt = torch.empty(max(n, 1), dtype=torch.float32, device=dev)
    own_ws = workspace is None
    workspace = _gdn_workspace(workspace, B, H, T, S, D, dev, "gdn_fwd")
    s = _stream(stream, dev)
    st = _call(dev, "gdn_fwd", _ptr(alpha), _ptr(b), _ptr(v), _ptr(c), _ptr(h0), _ptr(o), _ptr(ckpt),
                       B, H, T, S, D, _ptr(workspace),
                       workspace.numel() * workspace.element_size(), s)
    _check(st, "gdn_fwd")
    if own_ws:
        _release_after(workspace, s, dev)
    return o, ckpt


def gdn_workspace_bytes(B, H, T, S, D) -> int:
    return int(lib().gdn_workspace_bytes(B, H, T, S, D))


def _release_after(t, s, dev):
    """A scratch tensor allocated here and used by work queued on stream `s`:
    when `s` is not torch's current stream, tell the caching allocator not to
    reuse its memory before that work is done (it orders reuse by the
    allocation stream only)."""
    h = s.value or 0  # ctypes gives None for the null stream
    if h == torch.cuda.current_stream(dev).cuda_stream:
        return
    ds = torch.cuda.default_stream(dev)
    t.record_stream(ds if h == ds.cuda_stream else torch.cuda.ExternalStream(h, device=dev))


def _gdn_workspace(workspace, B, H, T, S, D, dev, name):
    nws = gdn_workspace_bytes(B, H, T, S, D)
    if workspace is None:
        return torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
    if not workspace.is_contiguous() or workspace.numel() * workspace.element_size() < nws:
        raise ValueError(f"{name} workspace must be a contiguous tensor of >= {nws} bytes")
    return workspace


def gdn_bwd(alpha, b, v, c, ckpt, dout, *, need_dh0=True, out=None, workspace=None,
            stream=None):
    """Backward of L = sum <dout_t, o_t>: returns (dalpha, db, dv, dc, dh0).

    workspace: a device tensor of at least gdn_workspace_bytes() bytes
    (allocated here when None)."""
    B, H, T, S, D = _gdn_dims(alpha, b, v, c)
    dev = alpha.device
    _need(dout, "dout", dtype=torch.float32, shape=(B, H, T, D), device=dev)
    if ckpt is None:
        raise ValueError("gdn_bwd needs the forward's checkpoint buffer")
    if out is not None:
        dal, db, dv, dc, dh0 = out
    else:
        dal, db, dv, dc = (torch.empty_like(t) for t in (alpha, b, v, c))
        dh0 = torch.empty((B, H, S, D), dtype=torch.float32, device=dev) if need_dh0 else None
    own_ws = workspace is None
    workspace = _gdn_workspace(workspace, B, H, T, S, D, dev, "gdn_bwd")
    s = _stream(stream, dev)
    st = _call(dev, "gdn_bwd", _ptr(alpha), _ptr(b), _ptr(v), _ptr(c), _ptr(ckpt), _ptr(dout), _ptr(dal),
                       _ptr(db), _ptr(dv), _ptr(dc), _ptr(dh0), B, H, T, S, D, _ptr(workspace),
                       workspace.numel() * workspace.element_size(), s)
    _check(st, "gdn_bwd")
    if own_ws:
        _release_after(workspace, s, dev)
    return dal, db, dv, dc, dh0


def scan_fwd_noalloc(a, x, h0=None, cu_seqlens=None, reverse=False, *, out=None, stream=None):
    """scan_fwd for callers that cannot allocate device memory.

    The scan's scratch is a fixed array inside libscan (no workspace, no
    allocation by the library). Only `out` is allocated here when not given;
    a caller that cannot allocate passes its own `out`. Overlapping calls on
    one GPU share that scratch and must be serialised; the first call on a
    device should come before any stream capture.
    """
    _need(a, "a")
    dev = a.device
    dt = _dtype_code(a)
    B, C, T, n = _scalar_dims(a, cu_seqlens)
    _need(x, "x", dtype=a.dtype, shape=a.shape, device=dev)
    _need(h0, "h0", dtype=torch.float32, shape=(n, C) if cu_seqlens is not None else (B, C),
          device=dev)
    h = out if out is not None else torch.empty(a.shape, dtype=torch.float32, device=dev)
    _need(h, "out", dtype=torch.float32, shape=a.shape, device=dev)
    st = _call(dev, "scan_fwd_noalloc", _ptr(a), _ptr(x), _ptr(h0), _ptr(cu_seqlens), n, _ptr(h), B, C, T,
                                dt, int(bool(reverse)), _stream(stream, dev))
    _check(st, "scan_fwd_noalloc")
    return h


def _rglru_args(x, gate_a, gate_x, a_param, segment_pos, h0):
    _need(x, "x")
    if x.dim() != 3:
        raise ValueError("x: expected [B, C, T]")
    dev = x.device
    B, C, T = x.shape
    _need(gate_a, "gate_a", dtype=x.dtype, shape=x.shape, device=dev)
    _need(gate_x, "gate_x", dtype=x.dtype, shape=x.shape, device=dev)
    _need(a_param, "a_param", dtype=torch.float32, shape=(C,), device=dev)
    _need(segment_pos, "segment_pos", dtype=torch.int32, shape=(B, T), device=dev)
    _need(h0, "h0", dtype=torch.float32, shape=(B, C), device=dev)
    return dev, B, C, T


def rglru_fwd(x, gate_a, gate_x, a_param, segment_pos=None, h0=None, *, out=None, stream=None):
    """RG-LRU gate preparation and scan: h_t = a_t h_{t-1} + sqrt(1 - a_t^2)
    sigmoid(gate_x_t) x_t, a_t = sigmoid(a_param)^(8 sigmoid(gate_a_t)), a reset
    where segment_pos == 0. x, gate_a, gate_x [B, C, T] fp32 or bf16; a_param
    [C]; segment_pos int32 [B, T] or None; h0 [B, C] or None. Returns h
    [B, C, T] (fp32)."""
    dev, B, C, T = _rglru_args(x, gate_a, gate_x, a_param, segment_pos, h0)
    dt = _dtype_code(x)
    h = out if out is not None else torch.empty(x.shape, dtype=torch.float32, device=dev)
    _need(h, "out", dtype=torch.float32, shape=x.shape, device=dev)
    st = _call(dev, "rglru_fwd", _ptr(x), _ptr(gate_a), _ptr(gate_x), _ptr(a_param),
               _ptr(segment_pos), _ptr(h0), _ptr(h), B, C, T, dt, _stream(stream, dev))
    _check(st, "rglru_fwd")
    return h


def rglru_bwd(x, gate_a, gate_x, a_param, h, dh, segment_pos=None, h0=None, *, out=None,
              stream=None, need_dh0=True):
    """Gradients of L = sum dh * h for h = rglru_fwd(...): (dx, dgate_a,
    dgate_x, da_param, dh0), the first three in x's dtype; dh0 is None when
    need_dh0 is False."""
    dev, B, C, T = _rglru_args(x, gate_a, gate_x, a_param, segment_pos, h0)
    dt = _dtype_code(x)
    _need(h, "h", dtype=torch.float32, shape=x.shape, device=dev)
    _need(dh, "dh", dtype=torch.float32, shape=x.shape, device=dev)
    if out is not None:
        dx, dga, dgx, dap, dh0 = out
    else:
        dx, dga, dgx = (torch.empty(x.shape, dtype=x.dtype, device=dev) for _ in range(3))
        dap = torch.empty(C, dtype=torch.float32, device=dev)
        dh0 = torch.empty(B, C, dtype=torch.float32, device=dev) if need_dh0 else None
    for t, name in ((dx, "dx"), (dga, "dgate_a"), (dgx, "dgate_x")):
        _need(t, name, dtype=x.dtype, shape=x.shape, device=dev)
    _need(dap, "da_param", dtype=torch.float32, shape=(C,), device=dev)
    _need(dh0, "dh0", dtype=torch.float32, shape=(B, C), device=dev)
    st = _call(dev, "rglru_bwd", _ptr(x), _ptr(gate_a), _ptr(gate_x), _ptr(a_param),
               _ptr(segment_pos), _ptr(h0), _ptr(h), _ptr(dh), _ptr(dx), _ptr(dga), _ptr(dgx),
               _ptr(dap), _ptr(dh0), B, C, T, dt, _stream(stream, dev))
    _check(st, "rglru_bwd")
    return dx, dga, dgx, dap, dh0


def scan_noalloc_device_status(device=None, stream=None) -> int:
    """Sticky device status of scan_fwd_noalloc's scratch on `device` (after
    synchronising `stream`); resets it. Allocates nothing."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    return int(_call(device, "scan_noalloc_device_status", _stream(stream, device)))


def scan_copy(src, dst, mode=SCAN_COPY_VEC, *, status=None, stream=None):
    """Copy the bytes of src into dst (same byte size) with one of the
    library's bandwidth-reference copies (SCAN_COPY_VEC or SCAN_COPY_TMA).
    status: optional CUDA int32 tensor of one element that a TMA wait which
    expires sets to SCAN_ERR_TIMEOUT. Returns dst."""
    _need(src, "src")
    dev = src.device
    _need(dst, "dst", device=dev)
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("scan_copy: src and dst differ in size")
    _need(status, "status", dtype=torch.int32, device=dev)
    st = _call(dev, "scan_copy", _ptr(src), _ptr(dst), nbytes, int(mode), _ptr(status),
               _stream(stream, dev))
    _check(st, "scan_copy")
    return dst
