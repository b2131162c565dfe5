"""The C ABI without a GPU: the library builds, loads and exports every entry
point that include/libscan.h declares, and host-side argument checks reject bad
input before anything is launched."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def built():
    from associative_affine_scan_gb300 import build_lib
    path = build_lib.build()
    return ctypes.CDLL(path)


def declared_functions():
    with open(os.path.join(ROOT, "include", "libscan.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("scan_fwd", "scan_bwd", "scan_bidir_fwd", "scan_bidir_bwd", "scan_log_fwd",
               "scan_log_bwd", "affine_scan_fwd", "affine_scan_bwd", "scan_workspace_bytes",
               "scan_workspace_init", "scan_get_device_status", "scan_status_string"):
        assert fn in names


def test_library_exports_every_declared_symbol(built):
    for name in declared_functions():
        assert hasattr(built, name), name


def test_binding_names_match_the_header():
    import associative_affine_scan_gb300 as scan
    for name in declared_functions():
        assert name in scan.EXPORTED
        assert callable(getattr(scan, name))


def test_status_strings_and_version():
    import associative_affine_scan_gb300 as scan
    assert scan.scan_version() == 1
    for code in range(8):
        assert scan.scan_status_string(code).startswith("SCAN_")


def test_workspace_sizes():
    import associative_affine_scan_gb300 as scan
    lookback = {"variant": scan.SCAN_VARIANT_LOOKBACK}
    # look-back: header + 16 bytes per (branch, row, chunk of 512)
    assert scan.scan_workspace_bytes(scan.SCAN_OP_FWD, 8, 1536, 4096, opts=lookback) == \
        256 + 12288 * 8 * 16
    assert scan.scan_workspace_bytes(scan.SCAN_OP_BIDIR_FWD, 1, 2048, 1000, opts=lookback) == \
        256 + 2 * 2048 * 2 * 16
    # stationary needs only the header; rows that fill the GPU choose it
    assert scan.scan_workspace_bytes(scan.SCAN_OP_FWD, 8, 1536, 4096,
                                     opts={"variant": scan.SCAN_VARIANT_STATIONARY}) == 256
    assert scan.scan_workspace_bytes(scan.SCAN_OP_FWD, 8, 1536, 4096) == 256
    # stationary rows cut into segments on request hand their end state on
    # through the workspace; unsegmented stationary needs only the header
    assert scan.scan_workspace_bytes(scan.SCAN_OP_FWD, 1, 2048, 100000,
                                     opts={"variant": scan.SCAN_VARIANT_STATIONARY,
                                           "segments": 5}) == 256 + 2048 * 5 * 16
    assert scan.scan_workspace_bytes(scan.SCAN_OP_FWD, 1, 2048, 100000,
                                     opts={"variant": scan.SCAN_VARIANT_STATIONARY}) == 256
    assert scan.scan_workspace_bytes(scan.SCAN_OP_FWD, 1, 2048, 100000,
                                     opts={"variant": scan.SCAN_VARIANT_STATIONARY,
                                           "segments": 1}) == 256
    # few rows (here 64) take the look-back
    assert scan.scan_workspace_bytes(scan.SCAN_OP_FWD, 1, 64, 100000) == \
        256 + 64 * ((100000 + 511) // 512) * 16
    # affine k=v=4: one 52-float record per (lane, chunk of 64 steps)
    assert scan.scan_workspace_bytes(scan.SCAN_OP_AFFINE_FWD, 8, 256, 4096, 4, 4) == \
        256 + 8 * 256 * 64 * 52 * 4
    assert scan.scan_workspace_bytes(scan.SCAN_OP_AFFINE_FWD, 8, 256, 4096, 3, 4) == 0
    # the rest of the envelope: k = 16, v = 1 records hold P (256), Q (16),
    # the inclusive state (16) and 2 flags, padded to 292 floats
    assert scan.scan_workspace_bytes(scan.SCAN_OP_AFFINE_BWD, 8, 256, 4096, 16, 1) == \
        256 + 8 * 256 * 64 * 292 * 4
    assert scan.scan_workspace_bytes(scan.SCAN_OP_AFFINE_FWD, 1, 4, 64, 32, 1) == 0
    # rejected arguments size to 0
    assert scan.scan_workspace_bytes(scan.SCAN_OP_FWD, -1, 4, 4) == 0
    assert scan.scan_workspace_bytes(scan.SCAN_OP_FWD, 1, 4, 4, opts={"chunk": 100}) == 0
    assert scan.scan_workspace_bytes(scan.SCAN_OP_FWD, 1, 4, 4, opts={"chunk": 1024}) == 0
    assert scan.scan_workspace_bytes(scan.SCAN_OP_FWD, 1, 4, 4, opts={"variant": 4}) == 0
    # the log-space backward plans like the other scalar calls
    assert scan.scan_workspace_bytes(scan.SCAN_OP_LOG_BWD, 1, 64, 100000) == \
        256 + 64 * ((100000 + 511) // 512) * 16
    assert scan.scan_workspace_bytes(scan.SCAN_OP_LOG_BWD, 8, 1536, 4096) == 256
    # the stream variant walks whole rows per warp: the header is all it needs
    stream = {"variant": scan.SCAN_VARIANT_STREAM}
    assert scan.scan_workspace_bytes(scan.SCAN_OP_BIDIR_FWD, 1, 2048, 275479, opts=stream) == 256
    assert scan.scan_workspace_bytes(scan.SCAN_OP_FWD, 1, 2048, 100000,
                                     opts=dict(stream, segments=4)) == 256
    for bad in (1, 17, -2):
        assert scan.scan_workspace_bytes(scan.SCAN_OP_FWD, 1, 4, 4,
                                         opts=dict(stream, stages=bad)) == 0


def _raw(name):
    import associative_affine_scan_gb300 as scan
    return getattr(scan.lib(), name)


def test_host_side_checks_need_no_gpu():
    import associative_affine_scan_gb300 as scan
    f = _raw("scan_fwd")
    fake = ctypes.c_void_p(0x1000)
    ws = ctypes.c_void_p(0x100000)
    # bad dtype
    assert f(fake, fake, None, None, 0, fake, 1, 1, 4, 7, 0, None, ws, 4096, None) == \
        scan.SCAN_ERR_INVALID_ARG
    # negative size
    assert f(fake, fake, None, None, 0, fake, 1, -1, 4, 0, 0, None, ws, 4096, None) == \
        scan.SCAN_ERR_INVALID_ARG
    # packed layout requires B == 1
    assert f(fake, fake, None, fake, 1, fake, 2, 1, 4, 0, 0, None, ws, 4096, None) == \
        scan.SCAN_ERR_INVALID_ARG
    # missing / short workspace
    assert f(fake, fake, None, None, 0, fake, 1, 4, 4096, 0, 0, None, None, 0, None) == \
        scan.SCAN_ERR_WORKSPACE
    assert f(fake, fake, None, None, 0, fake, 1, 4, 4096, 0, 0, None, ws, 300, None) == \
        scan.SCAN_ERR_WORKSPACE
    # malformed host copy of cu_seqlens
    opts = scan.ScanOpts()
    bad = (ctypes.c_int32 * 3)(0, 7, 5)
    opts.cu_seqlens_host = ctypes.cast(bad, ctypes.POINTER(ctypes.c_int32))
    assert f(fake, fake, None, fake, 2, fake, 1, 4, 5, 0, 0, ctypes.byref(opts), ws, 1 << 20,
             None) == scan.SCAN_ERR_INVALID_ARG
    # bad option values
    opts = scan.ScanOpts()
    for r in (99, 9, -1):  # rows per block: 1..8, 0 = planner
        opts.rows_per_cta = r
        assert f(fake, fake, None, None, 0, fake, 1, 4, 64, 0, 0, ctypes.byref(opts), ws, 1 << 20,
                 None) == scan.SCAN_ERR_INVALID_ARG
    # empty problem: nothing to launch, OK
    assert f(None, None, None, None, 0, None, 1, 0, 64, 0, 0, None, ws, 4096, None) == scan.SCAN_OK


def test_backward_log_bidir_affine_host_checks_need_no_gpu():
    """The other entry points reject malformed calls on the host too (bad
    dtype, negative size, missing workspace, a missing required pointer,
    misaligned block tensors), and an empty problem returns OK without a
    launch."""
    import associative_affine_scan_gb300 as scan
    fake = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1004)
    ws = ctypes.c_void_p(0x100000)
    big = 1 << 30
    OK, INV, WS, AL = (scan.SCAN_OK, scan.SCAN_ERR_INVALID_ARG, scan.SCAN_ERR_WORKSPACE,
                       scan.SCAN_ERR_ALIGNMENT)

    # scan_bwd(a, h, dh, h0, cu, n, da, dx, dh0, B, C, T, dt, reverse, opts, ws, nws, stream)
    bwd = _raw("scan_bwd")

    def b1(a=fake, da=fake, dims=(1, 4, 64), dt=0, w=ws, nw=big):
        return bwd(a, fake, fake, None, None, 0, da, fake, None, *dims, dt, 0, None, w, nw, None)

    assert b1(dt=5) == INV
    assert b1(dims=(1, -4, 64)) == INV
    assert b1(w=None) == WS
    assert b1(a=None) == INV
    assert b1(da=None) == INV
    assert b1(a=None, da=None, dims=(1, 4, 0)) == OK

    # scan_bidir_fwd(af, xf, ar, xr, h0f, h0r, cu, n, hf, hr, B, C, T, dt, opts, ws, nws, stream)
    bf = _raw("scan_bidir_fwd")
    assert bf(fake, fake, fake, fake, None, None, None, 0, fake, fake, 1, 4, 64, 9, None, ws,
              big, None) == INV
    assert bf(fake, fake, None, fake, None, None, None, 0, fake, fake, 1, 4, 64, 0, None, ws,
              big, None) == INV
    assert bf(fake, fake, fake, fake, None, None, None, 0, fake, fake, 1, 4, 64, 0, None, None,
              0, None) == WS
    # scan_bidir_bwd(af, hf, dhf, h0f, ar, hr, dhr, h0r, cu, n, daf, dxf, dh0f, dar, dxr, dh0r,
    #                B, C, T, dt, opts, ws, nws, stream)
    bb = _raw("scan_bidir_bwd")
    assert bb(fake, fake, fake, None, fake, fake, fake, None, None, 0, fake, fake, None, None,
              fake, None, 1, 4, 64, 0, None, ws, big, None) == INV  # dar missing
    assert bb(None, None, None, None, None, None, None, None, None, 0, None, None, None, None,
              None, None, 1, 0, 64, 0, None, ws, big, None) == OK

    # scan_log_fwd(la, lx, lh0, cu, n, h, B, C, T, reverse, opts, ws, nws, stream)
    lf = _raw("scan_log_fwd")
    assert lf(fake, fake, None, None, 0, None, 1, 4, 64, 0, None, ws, big, None) == INV
    assert lf(fake, fake, None, None, 0, fake, -1, 4, 64, 0, None, ws, big, None) == INV
    assert lf(fake, fake, None, None, 0, fake, 1, 4, 4096, 0, None, ws, 16, None) == WS
    # scan_log_bwd(la, lx, h, dh, lh0, cu, n, dla, dlx, dlh0, B, C, T, reverse, opts, ws, nws, s)
    lb = _raw("scan_log_bwd")
    assert lb(fake, fake, fake, fake, None, None, 0, fake, None, None, 1, 4, 64, 0, None, ws,
              big, None) == INV  # d log x missing
    assert lb(None, None, None, None, None, None, 0, None, None, None, 1, 4, 0, 0, None, ws,
              big, None) == OK

    # affine_scan_bwd(A, H, dH, h0, dA, dB, dh0, B, T, N, k, v, opts, ws, nws, stream)
    ab = _raw("affine_scan_bwd")
    assert ab(fake, fake, fake, None, fake, fake, None, 1, 64, 4, 4, 3, None, ws, big, None) == \
        scan.SCAN_ERR_UNSUPPORTED
    assert ab(fake, fake, fake, None, fake, fake, None, 1, 64, 4, 4, 4, None, None, 0, None) == WS
    assert ab(fake, fake, None, None, fake, fake, None, 1, 64, 4, 4, 4, None, ws, big, None) == INV
    assert ab(fake, fake, fake, None, odd, fake, None, 1, 64, 4, 4, 4, None, ws, big, None) == AL
    # affine_prefix_fwd(A, Abar, B, T, N, k, opts, ws, nws, stream)
    pf = _raw("affine_prefix_fwd")
    assert pf(fake, None, 1, 64, 4, 4, None, ws, big, None) == INV
    assert pf(odd, fake, 1, 64, 4, 4, None, ws, big, None) == AL
    assert pf(None, None, 1, 0, 4, 4, None, ws, big, None) == OK
    # affine_prefix_bwd(A, Abar, dAbar, dA, accumulate, B, T, N, k, opts, ws, nws, stream)
    pb = _raw("affine_prefix_bwd")
    assert pb(fake, fake, fake, None, 0, 1, 64, 4, 4, None, ws, big, None) == INV
    assert pb(fake, fake, fake, odd, 1, 1, 64, 4, 4, None, ws, big, None) == AL
    assert pb(fake, fake, fake, fake, 0, 1, 64, 4, 5, None, ws, big, None) == \
        scan.SCAN_ERR_UNSUPPORTED


def test_gdn_host_checks_need_no_gpu():
    """gdn_fwd / gdn_bwd reject malformed calls on the host (no launch, no GPU
    needed), and the checkpoint and workspace sizes follow their layouts."""
    import associative_affine_scan_gb300 as scan
    fwd, bwd = _raw("gdn_fwd"), _raw("gdn_bwd")
    fake = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1004)  # not 16-byte aligned
    ws = ctypes.c_void_p(0x100000)
    B, H, T, S, D = 2, 3, 130, 32, 16
    # one S x D state per 32 steps; the workspace holds one S x D matrix per
    # 32-step chunk and the chunks' gate products (padded to 4 floats)
    chunks = B * H * ((T + 31) // 32)
    assert scan.gdn_checkpoint_bytes(B, H, T, S, D) == 4 * chunks * S * D
    nws = scan.gdn_workspace_bytes(B, H, T, S, D)
    assert nws == 4 * (chunks * S * D + (chunks + 3) // 4 * 4)
    for s_, d_ in ((8, 16), (32, 64), (0, 16)):
        assert scan.gdn_workspace_bytes(B, H, T, s_, d_) == 0
        assert scan.gdn_checkpoint_bytes(B, H, T, s_, d_) == 0
    assert scan.gdn_workspace_bytes(-1, H, T, S, D) == 0

    def f(alpha=fake, b=fake, v=fake, c=fake, h0=None, o=fake, ck=fake, dims=(B, H, T, S, D),
          w=ws, nw=nws):
        return fwd(alpha, b, v, c, h0, o, ck, *dims, w, nw, None)

    assert f(dims=(B, H, T, 8, 16)) == scan.SCAN_ERR_UNSUPPORTED
    assert f(dims=(B, -1, T, S, D)) == scan.SCAN_ERR_INVALID_ARG
    assert f(alpha=None) == scan.SCAN_ERR_INVALID_ARG
    assert f(o=None) == scan.SCAN_ERR_INVALID_ARG
    assert f(b=odd) == scan.SCAN_ERR_ALIGNMENT
    assert f(h0=odd) == scan.SCAN_ERR_ALIGNMENT
    assert f(w=None) == scan.SCAN_ERR_WORKSPACE
    assert f(nw=nws - 16) == scan.SCAN_ERR_WORKSPACE
    assert f(w=odd) == scan.SCAN_ERR_WORKSPACE
    assert f(alpha=None, b=None, v=None, c=None, o=None, ck=None, dims=(B, H, 0, S, D)) == \
        scan.SCAN_OK  # empty: nothing to launch

    def g(ck=fake, dout=fake, db=fake, dh0=None, dims=(B, H, T, S, D), w=ws, nw=nws):
        return bwd(fake, fake, fake, fake, ck, dout, fake, db, fake, fake, dh0, *dims, w, nw, None)

    assert g(dims=(B, H, T, 16, 64)) == scan.SCAN_ERR_UNSUPPORTED
    assert g(dims=(-1, H, T, S, D)) == scan.SCAN_ERR_INVALID_ARG
    assert g(ck=None) == scan.SCAN_ERR_INVALID_ARG  # the forward's checkpoints are required
    assert g(dout=None) == scan.SCAN_ERR_INVALID_ARG
    assert g(db=odd) == scan.SCAN_ERR_ALIGNMENT
    assert g(dh0=odd) == scan.SCAN_ERR_ALIGNMENT
    assert g(w=None) == scan.SCAN_ERR_WORKSPACE
    assert g(nw=nws - 16) == scan.SCAN_ERR_WORKSPACE
    assert g(dims=(0, H, T, S, D)) == scan.SCAN_OK  # no heads: nothing to do
    assert g(dims=(B, H, 0, S, D)) == scan.SCAN_OK  # no steps and no dh0: nothing to write


def test_affine_envelope_rejected_on_host():
    import associative_affine_scan_gb300 as scan
    f = _raw("affine_scan_fwd")
    fake = ctypes.c_void_p(0x1000)
    ws = ctypes.c_void_p(0x100000)
    assert f(fake, fake, None, fake, 1, 8, 4, 3, 4, None, ws, 1 << 20, None) == \
        scan.SCAN_ERR_UNSUPPORTED


def test_step_host_argument_checks_need_no_gpu():
    """scan_step_host rejects malformed calls before touching the GPU."""
    import associative_affine_scan_gb300 as scan
    from associative_affine_scan_gb300._binding import DeviceIO, HostIO
    f = _raw("scan_step_host")
    fk = 0x1000
    full = dict(a=fk, x=fk, h0=None, dh=fk, h=fk, da=fk, dx=fk, dh0=None)
    hio, dio = HostIO(**full), DeviceIO(**full)
    ws = ctypes.c_void_p(0x100000)
    call = lambda h, d, B=1, C=4, T=64, dt=0, pieces=0, opts=None, w=ws, nw=4096: f(
        ctypes.byref(h) if h is not None else None, ctypes.byref(d) if d is not None else None,
        B, C, T, dt, pieces, ctypes.byref(opts) if opts is not None else None, w, nw, None)
    assert call(None, dio) == scan.SCAN_ERR_INVALID_ARG
    assert call(hio, None) == scan.SCAN_ERR_INVALID_ARG
    assert call(hio, dio, dt=7) == scan.SCAN_ERR_INVALID_ARG
    assert call(hio, dio, C=-1) == scan.SCAN_ERR_INVALID_ARG
    assert call(hio, dio, pieces=65) == scan.SCAN_ERR_INVALID_ARG
    # h0 on one side only
    assert call(HostIO(**dict(full, h0=fk)), dio) == scan.SCAN_ERR_INVALID_ARG
    assert call(hio, DeviceIO(**dict(full, dh0=fk))) == scan.SCAN_ERR_INVALID_ARG
    # a missing result buffer
    assert call(HostIO(**dict(full, dx=None)), dio) == scan.SCAN_ERR_INVALID_ARG
    # options and workspace are checked before the first copy is queued
    bad = scan.ScanOpts()
    bad.rows_per_cta = 99
    assert call(hio, dio, opts=bad) == scan.SCAN_ERR_INVALID_ARG
    bad = scan.ScanOpts()
    bad.chunk = 300
    assert call(hio, dio, opts=bad) == scan.SCAN_ERR_INVALID_ARG
    assert call(hio, dio, w=None) == scan.SCAN_ERR_WORKSPACE
    assert call(hio, dio, w=ctypes.c_void_p(0x100008)) == scan.SCAN_ERR_WORKSPACE
    lb = scan.ScanOpts()
    lb.variant = scan.SCAN_VARIANT_LOOKBACK  # per-chunk summaries: more than a header
    need = scan.scan_workspace_bytes(scan.SCAN_OP_FWD, 1, 4096, 4096, opts=lb)
    assert need > 4096
    assert call(hio, dio, C=8192, T=4096, pieces=2, opts=lb, nw=need - 16) == \
        scan.SCAN_ERR_WORKSPACE
    # empty problem: nothing to copy or launch
    assert call(HostIO(), DeviceIO(), C=0) == scan.SCAN_OK
    # valid calls pass those checks and reach the device: without a GPU the
    # first CUDA call fails (never run where a GPU would take the fake pointers)
    import torch
    if not torch.cuda.is_available():
        for opts in (None, lb):
            assert call(hio, dio, C=12288, T=4096, pieces=8, opts=opts, nw=1 << 30) == \
                scan.SCAN_ERR_CUDA


def test_copy_rejects_bad_arguments_on_the_host(built):
    """scan_copy checks mode, pointers and alignment before touching the GPU
    (the pointers here are placeholders that are never dereferenced)."""
    import associative_affine_scan_gb300 as scan
    f = scan.lib().scan_copy
    assert f(1024, 2048, 4096, 7, None, None) == scan.SCAN_ERR_INVALID_ARG
    assert f(None, 2048, 4096, scan.SCAN_COPY_VEC, None, None) == scan.SCAN_ERR_INVALID_ARG
    assert f(1024 + 4, 2048, 4096, scan.SCAN_COPY_VEC, None, None) == scan.SCAN_ERR_ALIGNMENT
    assert f(1024, 2048 + 8, 4096, scan.SCAN_COPY_TMA, None, None) == scan.SCAN_ERR_ALIGNMENT
    assert f(1024, 2048, 0, scan.SCAN_COPY_TMA, None, None) == scan.SCAN_OK


def test_rglru_rejects_bad_arguments_on_the_host(built):
    """rglru_fwd / rglru_bwd check sizes, dtype and required pointers before any
    CUDA call (the pointers here are placeholders that are never dereferenced)."""
    import associative_affine_scan_gb300 as scan
    L = scan.lib()
    p = 4096
    f32, bf16 = scan.SCAN_F32, scan.SCAN_BF16
    fwd, bwd = L.rglru_fwd, L.rglru_bwd
    assert fwd(p, p, p, p, None, None, p, -1, 2, 3, f32, None) == scan.SCAN_ERR_INVALID_ARG
    assert fwd(p, p, p, p, None, None, p, 1, 2, 3, 7, None) == scan.SCAN_ERR_INVALID_ARG
    assert fwd(p, p, p, p, None, None, p, 1, 2, 0, bf16, None) == scan.SCAN_OK  # nothing to do
    assert fwd(None, p, p, p, None, None, p, 1, 2, 3, f32, None) == scan.SCAN_ERR_INVALID_ARG
    assert fwd(p, p, p, None, None, None, p, 1, 2, 3, f32, None) == scan.SCAN_ERR_INVALID_ARG
    assert fwd(p, p, p, p, None, None, None, 1, 2, 3, f32, None) == scan.SCAN_ERR_INVALID_ARG
    assert fwd(p, p, p, p, None, None, p, 1, 1 << 31, 3, f32, None) == scan.SCAN_ERR_UNSUPPORTED
    args = [p] * 13
    assert bwd(*args, 1, 2, -3, f32, None) == scan.SCAN_ERR_INVALID_ARG
    assert bwd(*args, 1, 2, 3, 7, None) == scan.SCAN_ERR_INVALID_ARG
    assert bwd(*args, 1, 0, 3, f32, None) == scan.SCAN_OK  # no channels: nothing to write
    for i in (0, 1, 2, 3, 6, 7, 8, 9, 10, 11):  # the required pointers
        a = list(args)
        a[i] = None
        assert bwd(*a, 1, 2, 3, f32, None) == scan.SCAN_ERR_INVALID_ARG, i
