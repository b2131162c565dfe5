"""Guard bands around every output of every entry point.

Each output buffer handed to libscan is a view into the middle of a larger
buffer whose every word holds a sentinel bit pattern (a NaN with a payload no
kernel computes), with several KB on each side. After the call:

* every sentinel word outside the view is unchanged (no write past either end
  of the output, including the 16-byte vector stores at row and chunk edges,
  the row shifts of the 4-step groups and the tensor stores of the stream
  variant's tile rows);
* no sentinel word is left inside the view (every output element written);
* the values agree with the same call on plain buffers.

Views start 16-byte aligned (the vector and tensor-copy paths) and, where the
entry point accepts it, one element off (the scalar paths). Ragged T (1, 3,
127, 129, 4097), fp32 and bf16, dense and packed, every scalar variant, the
whole block envelope, the GDN chunk edges, the RG-LRU forward and backward and the
host-buffer step are covered (the entry point without allocation has its guard bands in
its own test file).
"""

import pytest
import torch

from associative_affine_scan_gb300 import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
PAD = 1024  # elements of sentinel on each side of every output
SENTINEL = {torch.float32: (torch.int32, 0x7FC0DEAD), torch.bfloat16: (torch.int16, 0x7FA5)}
TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-2}
# Outputs that are contractions of several fp32 results (the block form's dA
# and dh0, the outer-product state's gradients): two look-back runs compose
# earlier chunks in different orders, so two calls agree to their term scale,
# not to 1e-5 of the result; they are held to the 1e-3 gradient gate here (the
# parity tests check them against the oracle).
CONTRACTIONS = {"dA", "dh0", "dalpha", "db", "dv", "dc"}


class Guarded:
    """An output of `shape` and `dtype` inside a sentinel-filled buffer,
    starting `shift` elements past a 16-byte boundary."""

    def __init__(self, shape, dtype=torch.float32, shift=0, host=False):
        self.n = 1
        for s in shape:
            self.n *= int(s)
        self.lo = PAD + shift
        total = self.n + 2 * PAD + shift
        if host:
            self.buf = torch.empty(total, dtype=dtype, pin_memory=True)
        else:
            self.buf = torch.empty(total, dtype=dtype, device=DEV)
        itype, self.word = SENTINEL[dtype]
        self.bits = self.buf.view(itype)
        self.bits.fill_(self.word)
        self.t = self.buf[self.lo:self.lo + self.n].view(shape)

    def check(self, name):
        if not self.buf.is_cuda:
            torch.cuda.synchronize()
        bits = self.bits
        below = bits[:self.lo] != self.word
        above = bits[self.lo + self.n:] != self.word
        assert not bool(below.any()), f"{name}: {int(below.sum())} words written below the output"
        assert not bool(above.any()), f"{name}: {int(above.sum())} words written above the output"
        inside = bits[self.lo:self.lo + self.n] == self.word
        assert not bool(inside.any()), f"{name}: {int(inside.sum())} output words not written"


def close(got, ref, name, contraction=False):
    g, r = got.double().to(DEV), ref.double().to(DEV)
    if g.numel() == 0:
        return
    err = float(((g - r).abs() / r.abs().clamp_min(1.0)).max())
    tol = 1e-3 if contraction else TOL[got.dtype]
    assert err <= tol, (name, err)


def check_all(pairs, contractions=()):
    """pairs: (name, Guarded, reference tensor); names in `contractions` are
    compared at the gradient gate (see CONTRACTIONS)."""
    torch.cuda.synchronize()
    for name, gd, ref in pairs:
        gd.check(name)
        close(gd.t, ref, name, name in contractions)


def variants(lib):
    return [("planner", None),
            ("lookback", {"variant": lib.SCAN_VARIANT_LOOKBACK}),
            ("stationary", {"variant": lib.SCAN_VARIANT_STATIONARY}),
            ("segmented", {"variant": lib.SCAN_VARIANT_STATIONARY, "segments": 3}),
            ("stream", {"variant": lib.SCAN_VARIANT_STREAM}),
            ("stream_chunk_512", {"variant": lib.SCAN_VARIANT_STREAM, "chunk": 512})]


def packed_inputs(C, lens, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    T = int(cu[-1])
    a = torch.rand((C, T), generator=g)
    a[:, torch.rand(T, generator=g) < 0.01] = 0.0
    x = torch.randn((C, T), generator=g)
    dh = torch.randn((C, T), generator=g)
    h0 = torch.randn((len(lens), C), generator=g)
    return (a.to(dtype).to(DEV), x.to(dtype).to(DEV), dh.to(DEV), h0.to(DEV), cu.to(DEV))


def run_scalar(lib, a, x, dh, h0, cu, rev, opts, shift):
    dt = a.dtype
    n_h0 = tuple(h0.shape) if h0 is not None else (
        (cu.numel() - 1, a.shape[0]) if cu is not None else tuple(a.shape[:2]))
    ref_h = lib.scan_fwd(a, x, h0, cu, rev, opts=opts)
    ref_da, ref_dx, ref_dh0 = lib.scan_bwd(a, ref_h, dh, h0, cu, rev, opts=opts)
    h = Guarded(a.shape, torch.float32, shift)
    lib.scan_fwd(a, x, h0, cu, rev, out=h.t, opts=opts)
    da, dx = Guarded(a.shape, dt, shift), Guarded(a.shape, dt, shift)
    dh0 = Guarded(n_h0, torch.float32, 0)
    lib.scan_bwd(a, ref_h, dh, h0, cu, rev, out=(da.t, dx.t, dh0.t), opts=opts)
    check_all([("h", h, ref_h), ("da", da, ref_da), ("dx", dx, ref_dx), ("dh0", dh0, ref_dh0)])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [1, 3, 127, 129, 4097])
def test_guard_scalar_dense(lib, dtype, T):
    w = workloads.scalar_dense(2, 5, T, seed=T, h0=True, dtype=dtype)
    a, x, dh, h0 = w.a.to(DEV), w.x.to(DEV), w.dh.to(DEV), w.h0.to(DEV)
    for _, opts in variants(lib):
        for rev in (False, True):
            for shift in (0, 1):
                run_scalar(lib, a, x, dh, h0, None, rev, opts, shift)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_guard_scalar_many_rows(lib, dtype):
    """2100 rows: several blocks and row groups in every variant, a partial
    last group of rows, and the stream variant's rows dealt over its warps."""
    w = workloads.scalar_dense(3, 700, 1001, seed=4, h0=True, dtype=dtype)
    a, x, dh, h0 = w.a.to(DEV), w.x.to(DEV), w.dh.to(DEV), w.h0.to(DEV)
    for _, opts in variants(lib):
        for rev in (False, True):
            run_scalar(lib, a, x, dh, h0, None, rev, opts, 0)
    run_scalar(lib, a, x, dh, None, None, False, None, 1)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("lens", [[5, 0, 17, 1, 0, 300, 2, 129, 1000, 0], [4097], [1] * 40 + [513]])
def test_guard_scalar_packed(lib, dtype, lens):
    a, x, dh, h0, cu = packed_inputs(5, lens, seed=len(lens), dtype=dtype)
    for _, opts in variants(lib):
        for rev in (False, True):
            for shift in (0, 1):
                run_scalar(lib, a, x, dh, h0, cu, rev, opts, shift)
            run_scalar(lib, a, x, dh, None, cu, rev, opts, 0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_guard_bidir(lib, dtype):
    w = workloads.packed_bidir(seed=7, C=6, n_seqs=9, lo=1, hi=700, p_reset=0.01, dtype=dtype,
                               h0=True)
    af, xf, ar, xr, h0f, h0r, cu, dhf, dhr = (t.to(DEV) for t in (
        w.af, w.xf, w.ar, w.xr, w.h0f, w.h0r, w.cu_seqlens, w.dhf, w.dhr))
    for _, opts in variants(lib):
        for shift in (0, 1):
            rf, rr = lib.scan_bidir_fwd(af, xf, ar, xr, h0f, h0r, cu, opts=opts)
            hf, hr = Guarded(af.shape, torch.float32, shift), Guarded(af.shape, torch.float32, shift)
            lib.scan_bidir_fwd(af, xf, ar, xr, h0f, h0r, cu, out=(hf.t, hr.t), opts=opts)
            ref = lib.scan_bidir_bwd(af, rf, dhf, ar, rr, dhr, h0f, h0r, cu, opts=opts)
            outs = [Guarded(t.shape, t.dtype, shift if t.dim() == 2 and t.shape == af.shape else 0)
                    for t in ref]
            lib.scan_bidir_bwd(af, rf, dhf, ar, rr, dhr, h0f, h0r, cu,
                               out=tuple(g.t for g in outs), opts=opts)
            names = ("daf", "dxf", "dh0f", "dar", "dxr", "dh0r")
            check_all([("hf", hf, rf), ("hr", hr, rr)] + list(zip(names, outs, ref)))


@pytest.mark.parametrize("T", [1, 3, 127, 129, 4097])
def test_guard_log(lib, T):
    w = workloads.log_dense(2, 5, T, seed=T + 3, h0=True)
    la, lx, dh, lh0 = w.log_a.to(DEV), w.log_x.to(DEV), w.dh.to(DEV), w.log_h0.to(DEV)
    for _, opts in variants(lib):
        for rev in (False, True):
            for shift in (0, 1):
                ref_h = lib.scan_log_fwd(la, lx, lh0, None, rev, opts=opts)
                h = Guarded(la.shape, torch.float32, shift)
                lib.scan_log_fwd(la, lx, lh0, None, rev, out=h.t, opts=opts)
                ref = lib.scan_log_bwd(la, lx, ref_h, dh, lh0, None, rev, opts=opts)
                outs = (Guarded(la.shape, torch.float32, shift),
                        Guarded(la.shape, torch.float32, shift), Guarded(lh0.shape))
                lib.scan_log_bwd(la, lx, ref_h, dh, lh0, None, rev, out=tuple(g.t for g in outs),
                                 opts=opts)
                check_all([("h", h, ref_h)] +
                          list(zip(("dlog_a", "dlog_x", "dlog_h0"), outs, ref)))


def test_guard_log_packed(lib):
    a, x, dh, h0, cu = packed_inputs(3, [5, 0, 17, 1, 0, 300, 2, 129, 1000, 0], 9, torch.float32)
    la, lh0 = torch.log(a), torch.log(h0.abs() + 0.5)
    for _, opts in variants(lib):
        for rev in (False, True):
            ref_h = lib.scan_log_fwd(la, x, lh0, cu, rev, opts=opts)
            h = Guarded(la.shape, torch.float32, 1)
            lib.scan_log_fwd(la, x, lh0, cu, rev, out=h.t, opts=opts)
            ref = lib.scan_log_bwd(la, x, ref_h, dh, lh0, cu, rev, opts=opts)
            outs = (Guarded(la.shape), Guarded(la.shape), Guarded(lh0.shape))
            lib.scan_log_bwd(la, x, ref_h, dh, lh0, cu, rev, out=tuple(g.t for g in outs), opts=opts)
            check_all([("h", h, ref_h)] + list(zip(("dlog_a", "dlog_x", "dlog_h0"), outs, ref)))


def run_affine(lib, w, opts=None):
    A, Bm, dH = w.A.to(DEV), w.Bm.to(DEV), w.dH.to(DEV)
    h0 = w.h0.to(DEV) if w.h0 is not None else None
    ref_H = lib.affine_scan_fwd(A, Bm, h0, opts=opts)
    H = Guarded(Bm.shape)
    lib.affine_scan_fwd(A, Bm, h0, out=H.t, opts=opts)
    ref = lib.affine_scan_bwd(A, ref_H, dH, h0, opts=opts)
    outs = tuple(Guarded(t.shape) for t in ref)
    lib.affine_scan_bwd(A, ref_H, dH, h0, out=tuple(g.t for g in outs), opts=opts)
    check_all([("H", H, ref_H)] + list(zip(("dA", "dB", "dh0"), outs, ref)), CONTRACTIONS)


@pytest.mark.parametrize("k", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("v", [1, 2, 4, 8, 16])
def test_guard_affine_envelope(lib, k, v):
    w = workloads.affine(2, 131, 5, k, v, seed=k * 31 + v, h0=True)
    run_affine(lib, w)


@pytest.mark.parametrize("T", [1, 3, 127, 129, 4097])
def test_guard_affine_4x4(lib, T):
    w = workloads.affine(1, T, 37, 4, 4, seed=T, h0=True)
    run_affine(lib, w)
    run_affine(lib, w, {"chunk": 256})


@pytest.mark.parametrize("k", [1, 2, 4, 8, 16])
def test_guard_affine_prefix(lib, k):
    w = workloads.affine(2, 131, 5, k, k, seed=k + 5)
    A, dAbar = w.A.to(DEV), w.dH.to(DEV)
    ref = lib.affine_prefix_fwd(A)
    Abar = Guarded(A.shape)
    lib.affine_prefix_fwd(A, out=Abar.t)
    ref_dA = lib.affine_prefix_bwd(A, ref, dAbar)
    dA = Guarded(A.shape)
    lib.affine_prefix_bwd(A, ref, dAbar, dA.t)
    check_all([("Abar", Abar, ref), ("dA", dA, ref_dA)], CONTRACTIONS)


@pytest.mark.parametrize("S,D", [(16, 16), (16, 32), (32, 16), (32, 32)])
@pytest.mark.parametrize("T", [1, 31, 32, 33, 63, 64, 65, 97])
@pytest.mark.parametrize("heads", [(2, 3), (8, 20)])
def test_guard_gdn(lib, S, D, T, heads):
    B, H = heads
    w = workloads.gdn(B, H, T, S, D, seed=T + S + D, h0=True)
    alpha, b, v, c, dout, h0 = (t.to(DEV) for t in (w.alpha, w.b, w.v, w.c, w.dout, w.h0))
    ref_o, ref_ck = lib.gdn_fwd(alpha, b, v, c, h0)
    n_ck = lib.gdn_checkpoint_bytes(B, H, T, S, D) // 4
    o, ck = Guarded(ref_o.shape), Guarded((n_ck,))
    lib.gdn_fwd(alpha, b, v, c, h0, checkpoints=ck.t, out=o.t)
    ref = lib.gdn_bwd(alpha, b, v, c, ref_ck, dout)
    outs = tuple(Guarded(t.shape) for t in ref)
    lib.gdn_bwd(alpha, b, v, c, ref_ck, dout, out=tuple(g.t for g in outs))
    check_all([("o", o, ref_o), ("checkpoints", ck, ref_ck[:n_ck])] +
              list(zip(("dalpha", "db", "dv", "dc", "dh0"), outs, ref)), CONTRACTIONS)


@pytest.mark.parametrize("T", [1, 64, 65, 300])
@pytest.mark.parametrize("S,D", [(16, 32), (32, 32)])
def test_guard_gdn_workspace(lib, T, S, D):
    """Neither direction writes outside its gdn_workspace_bytes() bytes."""
    B, H = 2, 3
    w = workloads.gdn(B, H, T, S, D, seed=T + 8, h0=True)
    alpha, b, v, c, dout, h0 = (t.to(DEV) for t in (w.alpha, w.b, w.v, w.c, w.dout, w.h0))
    nb = lib.gdn_workspace_bytes(B, H, T, S, D)
    assert nb % 16 == 0
    ws = Guarded((nb // 4,))
    o, ck = lib.gdn_fwd(alpha, b, v, c, h0, workspace=ws.t.view(torch.uint8))
    lib.gdn_bwd(alpha, b, v, c, ck, dout, workspace=ws.t.view(torch.uint8))
    torch.cuda.synchronize()
    bits = ws.bits
    assert not bool((bits[:ws.lo] != ws.word).any()), "written below the workspace"
    assert not bool((bits[ws.lo + ws.n:] != ws.word).any()), "written above the workspace"


@pytest.mark.parametrize("T", [1, 3, 127, 128, 129, 4097])
@pytest.mark.parametrize("shift", [0, 1])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_guard_rglru(lib, T, shift, dtype):
    """The RG-LRU forward's h and the backward's dx, dgate_a, dgate_x (in the
    input dtype), da_param and dh0, 16-byte aligned (vector path) and one
    element off."""
    w = workloads.rglru(3, 5, T, seed=T + 3, docs=(1, 90), h0=True, dtype=dtype)
    x, ga, gx, ap, dh, seg, h0 = (t.to(DEV) for t in (w.x, w.gate_a, w.gate_x, w.a_param, w.dh,
                                                     w.segment_pos, w.h0))
    ref_h = lib.rglru_fwd(x, ga, gx, ap, seg, h0)
    ref = lib.rglru_bwd(x, ga, gx, ap, ref_h, dh, seg, h0)
    h = Guarded(x.shape, torch.float32, shift)
    lib.rglru_fwd(x, ga, gx, ap, seg, h0, out=h.t)
    outs = (Guarded(x.shape, dtype, shift), Guarded(x.shape, dtype, shift),
            Guarded(x.shape, dtype, shift), Guarded(ap.shape), Guarded(h0.shape))
    lib.rglru_bwd(x, ga, gx, ap, ref_h, dh, seg, h0, out=tuple(g.t for g in outs))
    check_all([("h", h, ref_h)] +
              list(zip(("dx", "dgate_a", "dgate_x", "da_param", "dh0"), outs, ref)))


@pytest.mark.parametrize("T,pieces", [(1000, 3), (1001, 4), (3, 2)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_guard_host_step(lib, T, pieces, dtype):
    """scan_step_host writes the device copies of its inputs, the device
    results and the host results: all of them guarded."""
    w = workloads.scalar_dense(2, 37, T, seed=T, h0=True, dtype=dtype)
    B, C = 2, 37
    pin = lambda t: t.contiguous().pin_memory()
    ha, hx, hdh, hh0 = pin(w.a), pin(w.x), pin(w.dh), pin(w.h0)
    o = lib.ScanOpts()
    o.variant = lib.SCAN_VARIANT_STATIONARY
    ref_h = lib.scan_fwd(w.a.to(DEV), w.x.to(DEV), w.h0.to(DEV), opts=o)
    ref_g = lib.scan_bwd(w.a.to(DEV), ref_h, w.dh.to(DEV), w.h0.to(DEV), opts=o)
    host = (Guarded((B, C, T), torch.float32, host=True), Guarded((B, C, T), dtype, host=True),
            Guarded((B, C, T), dtype, host=True), Guarded((B, C), torch.float32, host=True))
    dev = (Guarded((B, C, T), dtype), Guarded((B, C, T), dtype), Guarded((B, C)),
           Guarded((B, C, T)), Guarded((B, C, T)), Guarded((B, C, T), dtype),
           Guarded((B, C, T), dtype), Guarded((B, C)))
    lib.scan_step_host(ha, hx, hdh, hh0, out=tuple(g.t for g in host),
                       device=tuple(g.t for g in dev), pieces=pieces)
    torch.cuda.synchronize()
    check_all(list(zip(("host h", "host da", "host dx", "host dh0"), host,
                       (ref_h,) + tuple(ref_g))) +
              list(zip(("dev a", "dev x", "dev h0", "dev dh", "dev h", "dev da", "dev dx",
                        "dev dh0"), dev,
                       (w.a, w.x, w.h0, w.dh, ref_h) + tuple(ref_g))))
