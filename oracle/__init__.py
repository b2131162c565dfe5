"""Sequential fp64 CPU oracle for the associative affine scan.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the CUDA library and
its Python binding never do. It shares no code with the CUDA path: the
arithmetic lives in ``oracle.c`` (plain C, double precision, one left-to-right
loop per row, segment or lane), and this module only marshals numpy arrays.

What each routine follows (page titles and sections of the source pages):

* ``scan_fwd`` / ``scan_bwd``: "associative_scan_triton" README, quick start
  (h[t] = g[t] * h[t-1] + x[t], cu_seqlens packing, bidirectional branches) and
  how it works (reverse scan on shifted gates, d_gates = shifted_states *
  d_tokens).
* ``scan_log_fwd`` / ``scan_log_bwd``: "Triton scan kernels", One
  associative-scan family (the same recurrence carried in log space).
* ``affine_fwd`` / ``affine_bwd``: "Triton scan kernels", One associative-scan
  family, Kernel design, and Autograd integration and the reversed-scan
  backward (reverse scan with A_{t+1}^T).
* ``chunk_summary`` / ``compose``: "Our RG-LRU GPU audit", Exact real chunk
  algebra.
* ``gdn_fwd`` / ``gdn_bwd``: "Operations & Triton Kernels" (HyMo), The chunked
  GDN algorithm (write h_t = alpha_t h_{t-1} + b_t v_t^T, read o_t = c_t . h_t)
  and Mathematical Derivation of the Reverse-Time Backward Pass.
* ``rglru_fwd`` / ``rglru_bwd``: "Our RG-LRU GPU audit", Strengthened fused
  path (gate logits, a_param, segment_pos, initial state; the square-root
  multiplier and write; the clipped square-root backward) and Exact real chunk
  algebra (a reset is a_t = 0), with the method's own gate formulas, which the
  pages name but do not print (oracle.h states them).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain cc, no CUDA)."""
    stale = (not os.path.exists(_LIB) or
             os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["cc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            sig = {
                "oracle_scan_fwd": [_dp, _dp, _dp, _ip, ctypes.c_int, _dp, _i64, _i64, _i64, ctypes.c_int],
                "oracle_scan_bwd": [_dp, _dp, _dp, _ip, ctypes.c_int, _dp, _dp, _dp, _dp,
                                    _i64, _i64, _i64, ctypes.c_int],
                "oracle_scan_log_fwd": [_dp, _dp, _dp, _ip, ctypes.c_int, _dp, _i64, _i64, _i64,
                                        ctypes.c_int],
                "oracle_scan_log_bwd": [_dp, _dp, _dp, _ip, ctypes.c_int, _dp, _dp, _dp, _dp,
                                        _i64, _i64, _i64, ctypes.c_int],
                "oracle_affine_fwd": [_dp, _dp, _dp, _dp, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int],
                "oracle_affine_bwd": [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _i64, _i64, _i64,
                                      ctypes.c_int, ctypes.c_int],
                "oracle_gdn_fwd": [_dp, _dp, _dp, _dp, _dp, _dp, _i64, _i64, _i64, _i64, _i64],
                "oracle_gdn_bwd": [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                   _i64, _i64, _i64, _i64, _i64],
                "oracle_rglru_fwd": [_dp, _dp, _dp, _dp, _ip, _dp, _dp, _i64, _i64, _i64],
                "oracle_rglru_bwd": [_dp, _dp, _dp, _dp, _ip, _dp, _dp, _dp, _dp, _dp, _dp,
                                     _dp, _i64, _i64, _i64],
            }
            for name, args in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            lib.oracle_chunk_summary.argtypes = [_dp, _dp, _i64, _dp, _dp]
            lib.oracle_chunk_summary.restype = None
            lib.oracle_compose.argtypes = [ctypes.c_double] * 4 + [_dp, _dp]
            lib.oracle_compose.restype = None
            _lib = lib
    return _lib


def _f64(arr):
    if arr is None:
        return None
    if hasattr(arr, "detach"):  # torch tensor -> numpy, values converted exactly
        arr = arr.detach().cpu().double().numpy()
    return np.ascontiguousarray(arr, dtype=np.float64)


def _ptr(arr, typ=_dp):
    return None if arr is None else arr.ctypes.data_as(typ)


def _cu(cu_seqlens):
    if cu_seqlens is None:
        return None, 0
    if hasattr(cu_seqlens, "detach"):
        cu_seqlens = cu_seqlens.detach().cpu().numpy()
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    return cu, int(cu.shape[0]) - 1


def _scalar_dims(a, cu):
    if cu is None:
        if a.ndim != 3:
            raise ValueError("dense scalar scan expects [B, C, T]")
        return a.shape
    if a.ndim != 2:
        raise ValueError("packed scalar scan expects [C, T]")
    return (1,) + a.shape


def scan_fwd(a, x, h0=None, cu_seqlens=None, reverse=False):
    """h_t = a_t h_{t-1} + x_t (reverse: h_t = a_t h_{t+1} + x_t), fp64."""
    a, x, h0 = _f64(a), _f64(x), _f64(h0)
    cu, n = _cu(cu_seqlens)
    B, C, T = _scalar_dims(a, cu)
    h = np.empty_like(a)
    rc = _load().oracle_scan_fwd(_ptr(a), _ptr(x), _ptr(h0), _ptr(cu, _ip), n, _ptr(h),
                                 B, C, T, int(bool(reverse)))
    if rc:
        raise ValueError("oracle_scan_fwd: malformed arguments")
    return h


def scan_bwd(a, x, dh, h0=None, cu_seqlens=None, reverse=False):
    """Returns (da, dx, dh0) of L = sum dh * h; dh0 has h0's layout."""
    a, x, dh, h0 = _f64(a), _f64(x), _f64(dh), _f64(h0)
    cu, n = _cu(cu_seqlens)
    B, C, T = _scalar_dims(a, cu)
    da = np.empty_like(a)
    dx = np.empty_like(a)
    dh0 = np.empty((n, C) if cu is not None else (B, C), dtype=np.float64)
    rc = _load().oracle_scan_bwd(_ptr(a), _ptr(x), _ptr(h0), _ptr(cu, _ip), n, _ptr(dh),
                                 _ptr(da), _ptr(dx), _ptr(dh0), B, C, T, int(bool(reverse)))
    if rc:
        raise ValueError("oracle_scan_bwd: malformed arguments")
    return da, dx, dh0


def scan_log_fwd(log_a, log_x, log_h0=None, cu_seqlens=None, reverse=False):
    """h_t = exp(l_t), l_t = logaddexp(l_{t-1} + log_a_t, log_x_t), fp64."""
    la, lx, lh0 = _f64(log_a), _f64(log_x), _f64(log_h0)
    cu, n = _cu(cu_seqlens)
    B, C, T = _scalar_dims(la, cu)
    h = np.empty_like(la)
    rc = _load().oracle_scan_log_fwd(_ptr(la), _ptr(lx), _ptr(lh0), _ptr(cu, _ip), n, _ptr(h),
                                     B, C, T, int(bool(reverse)))
    if rc:
        raise ValueError("oracle_scan_log_fwd: malformed arguments")
    return h


def scan_log_bwd(log_a, log_x, dh, log_h0=None, cu_seqlens=None, reverse=False):
    """Returns (dlog_a, dlog_x, dlog_h0) of L = sum dh * h for the log-space scan."""
    la, lx, dh, lh0 = _f64(log_a), _f64(log_x), _f64(dh), _f64(log_h0)
    cu, n = _cu(cu_seqlens)
    B, C, T = _scalar_dims(la, cu)
    dla = np.empty_like(la)
    dlx = np.empty_like(la)
    dlh0 = np.empty((n, C) if cu is not None else (B, C), dtype=np.float64)
    rc = _load().oracle_scan_log_bwd(_ptr(la), _ptr(lx), _ptr(lh0), _ptr(cu, _ip), n, _ptr(dh),
                                     _ptr(dla), _ptr(dlx), _ptr(dlh0), B, C, T,
                                     int(bool(reverse)))
    if rc:
        raise ValueError("oracle_scan_log_bwd: malformed arguments")
    return dla, dlx, dlh0


def affine_fwd(A, Bm, h0=None):
    """H_t = A_t H_{t-1} + B_t; A [B,T,N,k,k], Bm [B,T,N,k,v], h0 [B,N,k,v]."""
    A, Bm, h0 = _f64(A), _f64(Bm), _f64(h0)
    B, T, N, k, _ = A.shape
    v = Bm.shape[-1]
    H = np.empty_like(Bm)
    rc = _load().oracle_affine_fwd(_ptr(A), _ptr(Bm), _ptr(h0), _ptr(H), B, T, N, k, v)
    if rc:
        raise ValueError("oracle_affine_fwd: malformed arguments")
    return H


def affine_bwd(A, Bm, dH, h0=None):
    """Returns (dA, dB, dh0) of L = sum <dH_t, H_t>."""
    A, Bm, dH, h0 = _f64(A), _f64(Bm), _f64(dH), _f64(h0)
    B, T, N, k, _ = A.shape
    v = Bm.shape[-1]
    dA = np.empty_like(A)
    dB = np.empty_like(Bm)
    dh0 = np.empty((B, N, k, v), dtype=np.float64)
    rc = _load().oracle_affine_bwd(_ptr(A), _ptr(Bm), _ptr(h0), _ptr(dH), _ptr(dA), _ptr(dB),
                                   _ptr(dh0), B, T, N, k, v)
    if rc:
        raise ValueError("oracle_affine_bwd: malformed arguments")
    return dA, dB, dh0


def gdn_fwd(alpha, b, v, c, h0=None):
    """o_t = h_t^T c_t with h_t = alpha_t h_{t-1} + b_t v_t^T ("Operations & Triton
    Kernels" (HyMo), The chunked GDN algorithm). alpha [B,H,T]; b, c [B,H,T,S];
    v [B,H,T,D]; h0 [B,H,S,D] or None. Returns o [B,H,T,D]."""
    alpha, b, v, c, h0 = _f64(alpha), _f64(b), _f64(v), _f64(c), _f64(h0)
    B, H, T, S = b.shape
    D = v.shape[-1]
    o = np.empty((B, H, T, D), dtype=np.float64)
    rc = _load().oracle_gdn_fwd(_ptr(alpha), _ptr(b), _ptr(v), _ptr(c), _ptr(h0), _ptr(o),
                                B, H, T, S, D)
    if rc:
        raise ValueError("oracle_gdn_fwd: malformed arguments")
    return o


def gdn_bwd(alpha, b, v, c, dout, h0=None):
    """Gradients of L = sum <dout_t, o_t>: (dalpha, db, dv, dc, dh0) (the same
    page, Mathematical Derivation of the Reverse-Time Backward Pass)."""
    alpha, b, v, c, dout, h0 = _f64(alpha), _f64(b), _f64(v), _f64(c), _f64(dout), _f64(h0)
    B, H, T, S = b.shape
    D = v.shape[-1]
    da = np.empty_like(alpha)
    db = np.empty_like(b)
    dv = np.empty_like(v)
    dc = np.empty_like(c)
    dh0 = np.empty((B, H, S, D), dtype=np.float64)
    rc = _load().oracle_gdn_bwd(_ptr(alpha), _ptr(b), _ptr(v), _ptr(c), _ptr(h0), _ptr(dout),
                                _ptr(da), _ptr(db), _ptr(dv), _ptr(dc), _ptr(dh0), B, H, T, S, D)
    if rc:
        raise ValueError("oracle_gdn_bwd: malformed arguments")
    return da, db, dv, dc, dh0


def _seg(segment_pos):
    if segment_pos is None:
        return None
    if hasattr(segment_pos, "detach"):
        segment_pos = segment_pos.detach().cpu().numpy()
    return np.ascontiguousarray(segment_pos, dtype=np.int32)


def rglru_fwd(x, gate_a, gate_x, a_param, segment_pos=None, h0=None):
    """h_t = a_t h_{t-1} + sqrt(1 - a_t^2) sigmoid(gate_x_t) x_t with
    a_t = sigmoid(a_param)^(8 sigmoid(gate_a_t)); a reset where segment_pos == 0.
    x, gate_a, gate_x [B, C, T]; a_param [C]; segment_pos [B, T] or None;
    h0 [B, C] or None. Returns h [B, C, T]."""
    x, ga, gx, ap, h0 = _f64(x), _f64(gate_a), _f64(gate_x), _f64(a_param), _f64(h0)
    seg = _seg(segment_pos)
    B, C, T = x.shape
    h = np.empty_like(x)
    rc = _load().oracle_rglru_fwd(_ptr(x), _ptr(ga), _ptr(gx), _ptr(ap), _ptr(seg, _ip),
                                  _ptr(h0), _ptr(h), B, C, T)
    if rc:
        raise ValueError("oracle_rglru_fwd: malformed arguments")
    return h


def rglru_bwd(x, gate_a, gate_x, a_param, dh, segment_pos=None, h0=None):
    """Gradients of L = sum dh * h: (dx, dgate_a, dgate_x, da_param, dh0)."""
    x, ga, gx, ap, dh, h0 = (_f64(x), _f64(gate_a), _f64(gate_x), _f64(a_param), _f64(dh),
                             _f64(h0))
    seg = _seg(segment_pos)
    B, C, T = x.shape
    dx, dga, dgx = np.empty_like(x), np.empty_like(x), np.empty_like(x)
    dap = np.empty(C, dtype=np.float64)
    dh0 = np.empty((B, C), dtype=np.float64)
    rc = _load().oracle_rglru_bwd(_ptr(x), _ptr(ga), _ptr(gx), _ptr(ap), _ptr(seg, _ip),
                                  _ptr(h0), _ptr(dh), _ptr(dx), _ptr(dga), _ptr(dgx), _ptr(dap),
                                  _ptr(dh0), B, C, T)
    if rc:
        raise ValueError("oracle_rglru_bwd: malformed arguments")
    return dx, dga, dgx, dap, dh0


def chunk_summary(a, x):
    """(P, Q) of a run of scalar steps, built left to right."""
    a, x = _f64(a), _f64(x)
    P, Q = ctypes.c_double(), ctypes.c_double()
    _load().oracle_chunk_summary(_ptr(a), _ptr(x), a.shape[0], ctypes.byref(P), ctypes.byref(Q))
    return P.value, Q.value


def compose(s1, s2):
    """Summary of "apply s1 then s2" for scalar summaries (P, Q)."""
    P, Q = ctypes.c_double(), ctypes.c_double()
    _load().oracle_compose(s1[0], s1[1], s2[0], s2[1], ctypes.byref(P), ctypes.byref(Q))
    return P.value, Q.value
