"""GPU parity of the scalar and log-space scans against the fp64 oracle.

Every call goes through the C ABI (the ctypes binding). Tolerances follow the
stated target: elementwise max |got - ref| / max(1, |ref|) <= 1e-5 for fp32
results and <= 1e-2 for results stored in bf16. Dyadic inputs (every partial
result exact in fp32) must match bit for bit, and so must everything that only
depends on cu_seqlens and reset indexing.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from _sweep import max_rel, sweep
from associative_affine_scan_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL32 = 1e-5
TOLBF = 1e-2
DEV = torch.device("cuda", 0)
HERE = os.path.dirname(os.path.abspath(__file__))


def rel_err(got, ref):
    if isinstance(got, torch.Tensor):
        got = got.detach().double().cpu().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref))))


def cuda(*ts):
    return [None if t is None else t.to(DEV) for t in ts]


def variants(scan):
    return [("lookback", {"variant": scan.SCAN_VARIANT_LOOKBACK}),
            ("stationary", {"variant": scan.SCAN_VARIANT_STATIONARY, "segments": 1}),
            ("segmented", {"variant": scan.SCAN_VARIANT_STATIONARY, "segments": 3}),
            ("stream", {"variant": scan.SCAN_VARIANT_STREAM}),
            ("stream_two_stages", {"variant": scan.SCAN_VARIANT_STREAM, "stages": 2})]


def check_fwd_bwd(scan, a, x, dh, h0=None, cu=None, reverse=False, opts=None, tol_h=TOL32,
                  tol_g=None):
    """Run fwd + bwd on the GPU and compare all outputs with the oracle."""
    tol_g = tol_g if tol_g is not None else (TOLBF if a.dtype == torch.bfloat16 else TOL32)
    ga, gx, gdh, gh0, gcu = cuda(a, x, dh, h0, cu)
    h = scan.scan_fwd(ga, gx, gh0, gcu, reverse, opts=opts)
    da, dx, dh0 = scan.scan_bwd(ga, h, gdh, gh0, gcu, reverse, opts=opts)
    torch.cuda.synchronize()
    assert scan.scan_get_device_status(DEV) == scan.SCAN_OK
    ref_h = oracle.scan_fwd(a, x, h0, cu, reverse)
    ref_da, ref_dx, ref_dh0 = oracle.scan_bwd(a, x, dh, h0, cu, reverse)
    errs = {"h": rel_err(h, ref_h), "da": rel_err(da, ref_da), "dx": rel_err(dx, ref_dx),
            "dh0": rel_err(dh0, ref_dh0)}
    assert errs["h"] <= tol_h, errs
    assert errs["da"] <= tol_g and errs["dx"] <= tol_g and errs["dh0"] <= TOL32, errs
    return h, da, dx, dh0


# ---------------------------------------------------------------------------
# dense layouts
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 3, 5, 127, 128, 129, 300, 511, 512, 513, 1029, 2053, 5000])
@pytest.mark.parametrize("reverse", [False, True])
def test_dense_fp32_shapes(lib, T, reverse):
    w = workloads.scalar_dense(2, 5, T, seed=T + 7 * reverse, h0=True)
    for _, opts in variants(lib):
        check_fwd_bwd(lib, w.a, w.x, w.dh, w.h0, None, reverse, opts)


@pytest.mark.parametrize("chunk", [128, 256, 512])
@pytest.mark.parametrize("rows_per_cta", [1, 3, 8])
def test_dense_chunk_and_rows(lib, chunk, rows_per_cta):
    w = workloads.scalar_dense(3, 7, 3001, seed=chunk + rows_per_cta, h0=True)
    for _, opts in variants(lib):
        o = dict(opts, chunk=chunk, rows_per_cta=rows_per_cta)
        check_fwd_bwd(lib, w.a, w.x, w.dh, w.h0, None, False, o)
        check_fwd_bwd(lib, w.a, w.x, w.dh, w.h0, None, True, o)


@pytest.mark.parametrize("T", [1, 130, 1027, 4096])
def test_dense_bf16(lib, T):
    w = workloads.scalar_dense(2, 6, T, seed=T, h0=True, dtype=torch.bfloat16)
    for _, opts in variants(lib):
        for rev in (False, True):
            check_fwd_bwd(lib, w.a, w.x, w.dh, w.h0, None, rev, opts)


@pytest.mark.parametrize("T", [128, 512, 2048, 8192])
def test_fp32_rmse_against_fp64(lib, T):
    """Accuracy level: root-mean-square error of the fp32 results against the
    fp64 oracle on the same fp32 inputs, C = 4 channels. The pages measure
    about 6.5e-8 for the forward ("associative_scan_triton" README, Numerical
    accuracy); fp32 rounding of one fused step per element, decaying with the
    gates, gives about 1e-7 here, and the bound sits ten times above that. The
    measured values are printed."""
    w = workloads.scalar_dense(1, 4, T, seed=T + 3, h0=False)
    a, x, dh = cuda(w.a, w.x, w.dh)
    h = lib.scan_fwd(a, x)
    da, dx, _ = lib.scan_bwd(a, h, dh)
    torch.cuda.synchronize()
    ref_h = oracle.scan_fwd(w.a, w.x)
    ref_da, ref_dx, _ = oracle.scan_bwd(w.a, w.x, w.dh)
    rmse = {}
    for name, got, ref in (("h", h, ref_h), ("dx", dx, ref_dx), ("da", da, ref_da)):
        diff = got.double().cpu().numpy() - np.asarray(ref, dtype=np.float64)
        rmse[name] = float(np.sqrt(np.mean(diff * diff)))
    print(f"T={T} rmse", rmse)
    assert all(v <= 1e-6 for v in rmse.values()), rmse


def test_dense_on_a_side_stream(lib):
    """A caller's own stream gets its own cached workspace and the results of
    the current stream: bit for bit when stationary; within the fp32 bound
    through the look-back, whose carry may be composed from predecessors'
    summaries in another order from run to run."""
    w = workloads.scalar_dense(2, 5, 3000, seed=21, h0=True)
    a, x, dh, h0 = cuda(w.a, w.x, w.dh, w.h0)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    for variant in (lib.SCAN_VARIANT_STATIONARY, lib.SCAN_VARIANT_LOOKBACK):
        opts = {"variant": variant}
        h_ref = lib.scan_fwd(a, x, h0, opts=opts)
        g_ref = lib.scan_bwd(a, h_ref, dh, h0, opts=opts)
        for _ in range(2):
            h = lib.scan_fwd(a, x, h0, opts=opts, stream=side)
            g = lib.scan_bwd(a, h, dh, h0, opts=opts, stream=side)
        side.synchronize()
        for got, ref in zip((h,) + tuple(g), (h_ref,) + tuple(g_ref)):
            if variant == lib.SCAN_VARIANT_STATIONARY:
                assert torch.equal(got, ref)
            else:
                assert rel_err(got, ref.double().cpu().numpy()) <= TOL32
    assert lib.scan_get_device_status(DEV, stream=side) == lib.SCAN_OK


def test_dense_no_h0_and_gates_near_one(lib):
    w = workloads.scalar_dense(2, 4, 4100, seed=3, gate="sigmoid2", h0=False)
    check_fwd_bwd(lib, w.a, w.x, w.dh, None, None, False)
    check_fwd_bwd(lib, w.a, w.x, w.dh, None, None, True)


def test_unaligned_pointers_take_the_scalar_path(lib):
    B, C, T = 2, 3, 517
    w = workloads.scalar_dense(B, C, T, seed=11, h0=True)
    n = B * C * T

    def shifted(t, dtype=torch.float32):
        buf = torch.zeros(n + 1, dtype=dtype, device=DEV)
        v = buf[1:].view(B, C, T)
        v.copy_(t.to(DEV))
        return v

    a, x, dh = shifted(w.a), shifted(w.x), shifted(w.dh)
    h = shifted(torch.zeros(B, C, T))
    lib.scan_fwd(a, x, w.h0.to(DEV), out=h)
    da = shifted(torch.zeros(B, C, T))
    dx = shifted(torch.zeros(B, C, T))
    dh0 = torch.empty(B, C, device=DEV)
    lib.scan_bwd(a, h, dh, w.h0.to(DEV), out=(da, dx, dh0))
    torch.cuda.synchronize()
    ref_h = oracle.scan_fwd(w.a, w.x, w.h0)
    ref = oracle.scan_bwd(w.a, w.x, w.dh, w.h0)
    assert rel_err(h, ref_h) <= TOL32
    assert rel_err(da, ref[0]) <= TOL32 and rel_err(dx, ref[1]) <= TOL32
    assert rel_err(dh0, ref[2]) <= TOL32


def test_single_sequence_config(lib):
    w = workloads.single_sequence(seed=0)
    check_fwd_bwd(lib, w.a, w.x, w.dh, None, w.cu_seqlens, False)
    # the same problem in the dense layout
    check_fwd_bwd(lib, w.a[None], w.x[None], w.dh[None], None, None, False)


# ---------------------------------------------------------------------------
# packed sequences, resets, bidirectional
# ---------------------------------------------------------------------------

def random_packed(C, lens, seed, dtype=torch.float32, h0=True, p_reset=0.0):
    g = torch.Generator().manual_seed(seed)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    T = int(cu[-1])
    a = torch.rand((C, T), generator=g)
    if p_reset:
        a[:, torch.rand(T, generator=g) < p_reset] = 0.0
    x = torch.randn((C, T), generator=g)
    dh = torch.randn((C, T), generator=g)
    hz = torch.randn((len(lens), C), generator=g) if h0 else None
    return a.to(dtype), x.to(dtype), dh, hz, cu


PACKED_LENS = [
    [5, 0, 17, 1, 0, 300, 2, 129, 1000, 0],
    [700],
    [0, 0, 3, 4096, 0, 1],
    [1] * 37 + [513, 2] + [0] * 5,
]


@pytest.mark.parametrize("case", range(len(PACKED_LENS)))
@pytest.mark.parametrize("C", [3, 5])
def test_packed_fp32(lib, case, C):
    a, x, dh, h0, cu = random_packed(C, PACKED_LENS[case], seed=case * 10 + C, p_reset=0.01)
    for _, opts in variants(lib):
        for chunk in (128, 512):
            o = dict(opts, chunk=chunk)
            for rev in (False, True):
                check_fwd_bwd(lib, a, x, dh, h0, cu, rev, o)
                check_fwd_bwd(lib, a, x, dh, None, cu, rev, o)


@pytest.mark.parametrize("case", range(len(PACKED_LENS)))
def test_packed_bf16(lib, case):
    a, x, dh, h0, cu = random_packed(4, PACKED_LENS[case], seed=case + 99, dtype=torch.bfloat16,
                                     p_reset=0.01)
    for _, opts in variants(lib):
        for rev in (False, True):
            check_fwd_bwd(lib, a, x, dh, h0, cu, rev, opts)


def test_packed_host_validation(lib):
    a, x, dh, h0, cu = random_packed(2, [3, 4], seed=1)
    bad = [0, 5, 4]
    with pytest.raises(lib.ScanError) as e:
        lib.scan_fwd(a.to(DEV), x.to(DEV), None, cu.to(DEV), opts={"cu_seqlens_host": bad})
    assert e.value.status == lib.SCAN_ERR_INVALID_ARG


def test_bidir_equals_two_single_branch_calls(lib):
    for dtype in (torch.float32, torch.bfloat16):
        w = workloads.packed_bidir(seed=5, C=6, n_seqs=9, lo=1, hi=700, p_reset=0.01, dtype=dtype,
                                   h0=True)
        g = cuda(w.af, w.xf, w.ar, w.xr, w.h0f, w.h0r, w.cu_seqlens, w.dhf, w.dhr)
        af, xf, ar, xr, h0f, h0r, cu, dhf, dhr = g
        for _, opts in variants(lib):
            hf, hr = lib.scan_bidir_fwd(af, xf, ar, xr, h0f, h0r, cu, opts=opts)
            hf1 = lib.scan_fwd(af, xf, h0f, cu, False, opts=opts)
            hr1 = lib.scan_fwd(ar, xr, h0r, cu, True, opts=opts)
            assert torch.equal(hf, hf1) and torch.equal(hr, hr1)
            grads = lib.scan_bidir_bwd(af, hf, dhf, ar, hr, dhr, h0f, h0r, cu, opts=opts)
            gf = lib.scan_bwd(af, hf, dhf, h0f, cu, False, opts=opts)
            gr = lib.scan_bwd(ar, hr, dhr, h0r, cu, True, opts=opts)
            for got, ref in zip(grads, gf + gr):
                assert torch.equal(got, ref)
            torch.cuda.synchronize()
            ref_hf = oracle.scan_fwd(w.af, w.xf, w.h0f, w.cu_seqlens, False)
            ref_hr = oracle.scan_fwd(w.ar, w.xr, w.h0r, w.cu_seqlens, True)
            assert rel_err(hf, ref_hf) <= TOL32 and rel_err(hr, ref_hr) <= TOL32


def dyadic(shape, seed):
    g = np.random.default_rng(seed)
    a = g.choice([0.0, 1.0, -1.0, 0.5, 1.0, 0.0, -1.0, 1.0], size=shape)
    x = g.integers(-4, 5, size=shape).astype(np.float64)
    dh = g.integers(-3, 4, size=shape).astype(np.float64)
    return a, x, dh


@pytest.mark.parametrize("packed", [False, True])
def test_dyadic_inputs_are_bit_exact(lib, packed):
    if packed:
        lens = [7, 0, 130, 1, 600, 0, 2000, 3]
        cu = np.zeros(len(lens) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lens)
        a, x, dh = dyadic((5, int(cu[-1])), 3)
        h0 = np.random.default_rng(4).integers(-3, 4, size=(len(lens), 5)).astype(np.float64)
        cu_t = torch.from_numpy(cu)
    else:
        a, x, dh = dyadic((2, 3, 2741), 5)
        h0 = np.random.default_rng(6).integers(-3, 4, size=(2, 3)).astype(np.float64)
        cu, cu_t = None, None
    ta, tx, tdh, th0 = (torch.from_numpy(v).float() for v in (a, x, dh, h0))
    for _, opts in variants(lib):
        for chunk in (128, 512):
            for rev in (False, True):
                o = dict(opts, chunk=chunk)
                ga, gx, gdh, gh0, gcu = cuda(ta, tx, tdh, th0, cu_t)
                h = lib.scan_fwd(ga, gx, gh0, gcu, rev, opts=o)
                da, dx, dh0 = lib.scan_bwd(ga, h, gdh, gh0, gcu, rev, opts=o)
                ref_h = oracle.scan_fwd(a, x, h0, cu, rev)
                ref_da, ref_dx, ref_dh0 = oracle.scan_bwd(a, x, dh, h0, cu, rev)
                assert np.array_equal(h.cpu().double().numpy(), ref_h)
                assert np.array_equal(dx.cpu().double().numpy(), ref_dx)
                assert np.array_equal(dh0.cpu().double().numpy(), ref_dh0)
                # da = g * h_prev is one rounding of an exact product
                assert np.array_equal(da.cpu().numpy(), ref_da.astype(np.float32))


@pytest.mark.parametrize("name", ["scalar_dense_dyadic.json", "scalar_packed_dyadic.json"])
def test_golden_worked_examples_bit_exact(lib, name):
    with open(os.path.join(HERE, "golden", name)) as f:
        g = json.load(f)
    cu = torch.tensor(g["cu_seqlens"], dtype=torch.int32) if "cu_seqlens" in g else None
    a, x, dh, h0 = (torch.tensor(g[k], dtype=torch.float32) for k in ("a", "x", "dh", "h0"))
    for key, rev in (("causal", False), ("reverse", True)):
        ga, gx, gdh, gh0, gcu = cuda(a, x, dh, h0, cu)
        h = lib.scan_fwd(ga, gx, gh0, gcu, rev)
        da, dx, dh0 = lib.scan_bwd(ga, h, gdh, gh0, gcu, rev)
        ref = g[key]
        assert h.cpu().tolist() == ref["h"]
        assert dx.cpu().tolist() == ref["dx"]
        assert dh0.cpu().tolist() == ref["dh0"]
        assert np.array_equal(da.cpu().numpy(), np.array(ref["da"], dtype=np.float32))


def test_segments_are_isolated(lib):
    a, x, dh, h0, cu = random_packed(4, [100, 0, 700, 33, 900], seed=8, p_reset=0.0)
    ga, gx, gdh, gh0, gcu = cuda(a, x, dh, h0, cu)
    for rev in (False, True):
        h = lib.scan_fwd(ga, gx, gh0, gcu, rev)
        g1 = lib.scan_bwd(ga, h, gdh, gh0, gcu, rev)
        a2, x2 = a.clone(), x.clone()
        a2[:, 100:800] = torch.rand(4, 700)
        x2[:, 100:800] = torch.randn(4, 700)
        ga2, gx2 = cuda(a2, x2)
        h2 = lib.scan_fwd(ga2, gx2, gh0, gcu, rev)
        g2 = lib.scan_bwd(ga2, h2, gdh, gh0, gcu, rev)
        keep = torch.cat([torch.arange(0, 100), torch.arange(800, a.shape[1])]).to(DEV)
        assert torch.equal(h[:, keep], h2[:, keep])
        for u, v in zip(g1[:2], g2[:2]):
            assert torch.equal(u[:, keep], v[:, keep])
        # dh0 rows of the untouched sequences are identical too
        assert torch.equal(g1[2][[0, 1, 3, 4]], g2[2][[0, 1, 3, 4]])


def test_resets_reproduce_x_exactly(lib):
    w = workloads.scalar_dense(2, 3, 3333, seed=12, h0=True)
    a = w.a.clone()
    a[..., ::97] = 0.0
    ga, gx, gh0 = cuda(a, w.x, w.h0)
    for rev in (False, True):
        h = lib.scan_fwd(ga, gx, gh0, None, rev)
        assert torch.equal(h[..., ::97], gx[..., ::97])


def test_stream_continuation(lib):
    w = workloads.scalar_dense(2, 4, 3000, seed=13, h0=True)
    ga, gx, gh0 = cuda(w.a, w.x, w.h0)
    whole = lib.scan_fwd(ga, gx, gh0)
    first = lib.scan_fwd(ga[..., :1234].contiguous(), gx[..., :1234].contiguous(), gh0)
    second = lib.scan_fwd(ga[..., 1234:].contiguous(), gx[..., 1234:].contiguous(),
                          first[..., -1].contiguous())
    torch.cuda.synchronize()
    ref = oracle.scan_fwd(w.a, w.x, w.h0)
    assert rel_err(torch.cat([first, second], -1), ref) <= TOL32
    assert rel_err(whole, ref) <= TOL32


def test_lookback_wait_limit_reports_timeout(lib):
    w = workloads.scalar_dense(1, 2, 4096, seed=14, h0=True)
    ga, gx, gh0 = cuda(w.a, w.x, w.h0)
    lib.scan_get_device_status(DEV)  # clear
    opts = {"variant": lib.SCAN_VARIANT_LOOKBACK, "chunk": 512, "test_stall": 1,
            "wait_limit_s": 1e-3}
    lib.scan_fwd(ga, gx, gh0, opts=opts)
    assert lib.scan_get_device_status(DEV) == lib.SCAN_ERR_TIMEOUT
    # the status was reset and the context still works
    h = lib.scan_fwd(ga, gx, gh0, opts={"variant": lib.SCAN_VARIANT_LOOKBACK, "chunk": 512})
    assert lib.scan_get_device_status(DEV) == lib.SCAN_OK
    assert rel_err(h, oracle.scan_fwd(w.a, w.x, w.h0)) <= TOL32


def test_lookback_records_cleared_before_tags_repeat(lib):
    """Record tags keep the launch epoch's low 30 bits, so on one workspace a
    tag comes back every 2^30 launches. The launch that ends just before the
    wrap must zero every record byte used on the workspace so far: set the
    epoch to 2^30 - 1, fill the records of an earlier, larger launch with
    words carrying the tag that epoch 2^30 will use, run a smaller launch,
    and check that all of them are zero afterwards and that both launches
    give the oracle's results."""
    import ctypes
    import struct
    from associative_affine_scan_gb300 import _binding
    big = workloads.scalar_dense(2, 64, 4096, seed=40, h0=True)
    small = workloads.scalar_dense(1, 4, 1000, seed=41, h0=True)
    opts = {"variant": lib.SCAN_VARIANT_LOOKBACK, "chunk": 512}
    a, x, h0 = cuda(big.a, big.x, big.h0)
    sa, sx, sh0 = cuda(small.a, small.x, small.h0)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    lib.scan_fwd(a, x, h0, opts=opts, stream=side)
    side.synchronize()
    ws = _binding._ws.current(DEV, ctypes.c_void_p(side.cuda_stream))
    words = ws.view(torch.int64)
    rec_words = 2 * 128 * 8  # 128 rows x 8 chunks of 512 steps, 16 bytes each
    stale_tag_inc = 2  # (2^30 << 2) | 2 in 32 bits
    huge = struct.unpack("<I", struct.pack("<f", 1e30))[0]
    words[0] = (2 ** 30 - 1) << 32  # ticket 0, epoch 2^30 - 1
    words[32:32 + rec_words] = (stale_tag_inc << 32) | huge
    torch.cuda.synchronize()
    hs = lib.scan_fwd(sa, sx, sh0, opts=opts, stream=side)
    side.synchronize()
    assert int(words[0]) == (2 ** 30) << 32
    assert int((words[32:32 + rec_words] != 0).sum()) == 0
    hb = lib.scan_fwd(a, x, h0, opts=opts, stream=side)
    side.synchronize()
    assert lib.scan_get_device_status(DEV, stream=side) == lib.SCAN_OK
    assert rel_err(hs, oracle.scan_fwd(small.a, small.x, small.h0)) <= TOL32
    assert rel_err(hb, oracle.scan_fwd(big.a, big.x, big.h0)) <= TOL32


def test_empty_inputs(lib):
    a = torch.empty(2, 3, 0, device=DEV)
    h = lib.scan_fwd(a, a)
    assert h.shape == (2, 3, 0)
    da, dx, dh0 = lib.scan_bwd(a, h, h, None)
    torch.cuda.synchronize()
    assert torch.equal(dh0, torch.zeros(2, 3, device=DEV))
    cu = torch.zeros(4, dtype=torch.int32, device=DEV)
    e = torch.empty(3, 0, device=DEV)
    _, _, dh0 = lib.scan_bwd(e, e, e, torch.ones(3, 3, device=DEV), cu)
    assert torch.equal(dh0, torch.zeros(3, 3, device=DEV))


# ---------------------------------------------------------------------------
# log space
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 5, 128, 129, 777, 4096])
@pytest.mark.parametrize("reverse", [False, True])
def test_log_dense(lib, T, reverse):
    w = workloads.log_dense(2, 3, T, seed=T, h0=True)
    for _, opts in variants(lib):
        for h0 in (w.log_h0, None):
            ga, gx, gh0 = cuda(w.log_a, w.log_x, h0)
            h = lib.scan_log_fwd(ga, gx, gh0, None, reverse, opts=opts)
            torch.cuda.synchronize()
            ref = oracle.scan_log_fwd(w.log_a, w.log_x, h0, None, reverse)
            assert rel_err(h, ref) <= TOL32


@pytest.mark.parametrize("reverse", [False, True])
def test_log_dense_infinities_and_wide_range(lib, reverse):
    """Dense rows whose runs hold log a = -inf (resets), log x = -inf (zero
    inputs), whole stretches with no mass at all, and log x over +-20 (terms
    that differ by up to e^40 inside one run)."""
    g = torch.Generator().manual_seed(77)
    B, C, T = 2, 5, 2048 + 37
    la = torch.nn.functional.logsigmoid(torch.randn((B, C, T), generator=g))
    lx = (8.0 * torch.randn((B, C, T), generator=g)).clamp(-20.0, 20.0)
    la[torch.rand((B, C, T), generator=g) < 0.02] = -math.inf
    lx[torch.rand((B, C, T), generator=g) < 0.05] = -math.inf
    la[:, 1, 300:700] = -math.inf  # every run here: no carried mass
    lx[:, 1, 300:700] = -math.inf  # and none added
    lx[:, 2, :600] = -math.inf     # rows that start empty
    lh0 = torch.randn((B, C), generator=g)
    lh0[0, 2] = -math.inf
    for _, opts in variants(lib):
        for h0 in (lh0, None):
            ga, gx, gh0 = cuda(la, lx, h0)
            h = lib.scan_log_fwd(ga, gx, gh0, None, reverse, opts=opts)
            torch.cuda.synchronize()
            ref = oracle.scan_log_fwd(la, lx, h0, None, reverse)
            assert torch.isfinite(h).all()
            assert rel_err(h, ref) <= TOL32


def test_log_packed_with_resets(lib):
    a, x, dh, h0, cu = random_packed(3, PACKED_LENS[0], seed=21, p_reset=0.02)
    la = torch.log(a)  # exact zeros become -inf
    for _, opts in variants(lib):
        for rev in (False, True):
            ga, gx, gh0, gcu = cuda(la, x, h0, cu)
            h = lib.scan_log_fwd(ga, gx, gh0, gcu, rev, opts=opts)
            torch.cuda.synchronize()
            ref = oracle.scan_log_fwd(la, x, h0, cu, rev)
            assert rel_err(h, ref) <= TOL32


def check_log_bwd(scan, la, lx, dh, lh0=None, cu=None, reverse=False, opts=None):
    """Log-space forward on the GPU, then its backward, against the oracle."""
    ga, gx, gdh, gh0, gcu = cuda(la, lx, dh, lh0, cu)
    h = scan.scan_log_fwd(ga, gx, gh0, gcu, reverse, opts=opts)
    dla, dlx, dlh0 = scan.scan_log_bwd(ga, gx, h, gdh, gh0, gcu, reverse, opts=opts)
    torch.cuda.synchronize()
    assert scan.scan_get_device_status(DEV) == scan.SCAN_OK
    ref = oracle.scan_log_bwd(la, lx, dh, lh0, cu, reverse)
    errs = (rel_err(dla, ref[0]), rel_err(dlx, ref[1]), rel_err(dlh0, ref[2]))
    assert all(e <= TOL32 for e in errs), errs


@pytest.mark.parametrize("T", [1, 5, 128, 129, 777, 4096])
@pytest.mark.parametrize("reverse", [False, True])
def test_log_bwd_dense(lib, T, reverse):
    w = workloads.log_dense(2, 3, T, seed=T + 1, h0=True)
    for _, opts in variants(lib):
        for h0 in (w.log_h0, None):
            check_log_bwd(lib, w.log_a, w.log_x, w.dh, h0, None, reverse, opts)


def test_log_bwd_packed_with_resets(lib):
    a, x, dh, h0, cu = random_packed(3, PACKED_LENS[0], seed=23, p_reset=0.02)
    la = torch.log(a)  # exact zeros become -inf
    lh0 = torch.log(h0.abs() + 0.5)
    for _, opts in variants(lib):
        for rev in (False, True):
            check_log_bwd(lib, la, x, dh, lh0, cu, rev, opts)


# ---------------------------------------------------------------------------
# full-size workloads in the benchmark's launch configuration
# ---------------------------------------------------------------------------

def test_full_dense_4k(lib):
    """Every output of the 8 x 1536 x 4096 workload, with the planner's choice
    and with each register-carry and stream scheme (the stream grid deals
    several rows to each warp at this size)."""
    w = workloads.dense_4k(seed=0)
    ref_h = oracle.scan_fwd(w.a, w.x, w.h0)
    ref_da, ref_dx, ref_dh0 = oracle.scan_bwd(w.a, w.x, w.dh, w.h0)
    ga, gx, gdh, gh0 = cuda(w.a, w.x, w.dh, w.h0)
    for opts in (None, {"variant": lib.SCAN_VARIANT_STATIONARY},
                 {"variant": lib.SCAN_VARIANT_STREAM},
                 {"variant": lib.SCAN_VARIANT_STREAM, "chunk": 256}):
        h = lib.scan_fwd(ga, gx, gh0, opts=opts)
        da, dx, dh0 = lib.scan_bwd(ga, h, gdh, gh0, opts=opts)
        torch.cuda.synchronize()
        assert lib.scan_get_device_status(DEV) == lib.SCAN_OK
        errs = (rel_err(h, ref_h), rel_err(da, ref_da), rel_err(dx, ref_dx),
                rel_err(dh0, ref_dh0))
        assert all(e <= TOL32 for e in errs), (opts, errs)
        del h, da, dx, dh0


def test_full_dense_64k_all_rows(lib):
    """Every output of the 8 x 1536 x 65536 workload (805 M elements per
    tensor) in the planner's launch configuration, against the oracle row by
    row (batches of rows on the host cores)."""
    w = workloads.dense_64k(seed=0)
    B, C, T = w.a.shape
    ga, gx, gdh = cuda(w.a, w.x, w.dh)
    h = lib.scan_fwd(ga, gx)
    da, dx, dh0 = lib.scan_bwd(ga, h, gdh, None)
    torch.cuda.synchronize()
    assert lib.scan_get_device_status(DEV) == lib.SCAN_OK
    del ga, gx, gdh
    a2, x2, dh2 = (t.view(B * C, T) for t in (w.a, w.x, w.dh))
    h2, da2, dx2 = (t.view(B * C, T) for t in (h, da, dx))
    dh0f = dh0.view(-1).cpu()

    def check(r0, r1):
        ra, rx, rdh = a2[r0:r1][None], x2[r0:r1][None], dh2[r0:r1][None]
        ref_h = oracle.scan_fwd(ra, rx)
        ref_da, ref_dx, ref_dh0 = oracle.scan_bwd(ra, rx, rdh)
        return {"h": max_rel(h2[r0:r1], ref_h[0]), "da": max_rel(da2[r0:r1], ref_da[0]),
                "dx": max_rel(dx2[r0:r1], ref_dx[0]), "dh0": max_rel(dh0f[r0:r1], ref_dh0[0])}

    errs = sweep(B * C, 96, check)
    print("dense_64k all rows", errs)
    assert errs["items"] == B * C
    assert all(errs[k] <= TOL32 for k in ("h", "da", "dx", "dh0")), errs


@pytest.mark.parametrize("variant", ["planner", "stream"])
def test_beyond_int32_elements_sampled_rows(lib, variant):
    """2^31 + 2,097,152 elements: every offset past element 2^31 needs 64-bit
    indexing. Rows on both sides of the boundary against the oracle."""
    if torch.cuda.get_device_properties(DEV).total_memory < (64 << 30):
        pytest.skip("needs about 52 GB of device memory")
    w = workloads.dense_beyond_int32(DEV, seed=0)
    B, C, T = w.a.shape
    assert B * C * T > 2 ** 31
    opts = {"variant": lib.SCAN_VARIANT_STREAM} if variant == "stream" else None
    h = lib.scan_fwd(w.a, w.x, w.h0, opts=opts)
    da, dx, dh0 = lib.scan_bwd(w.a, h, w.dh, w.h0, opts=opts)
    torch.cuda.synchronize()
    assert lib.scan_get_device_status(DEV) == lib.SCAN_OK
    first_past = 2 ** 31 // T  # 8192: the first row that starts past element 2^31
    for r in (0, 1, first_past - 1, first_past, C - 2, C - 1):
        ra, rx, rdh = (t[0, r][None, None].cpu() for t in (w.a, w.x, w.dh))
        rh0 = w.h0[:, r:r + 1].cpu()
        ref_h = oracle.scan_fwd(ra, rx, rh0)
        ref_da, ref_dx, ref_dh0 = oracle.scan_bwd(ra, rx, rdh, rh0)
        assert rel_err(h[0, r], ref_h[0, 0]) <= TOL32, r
        assert rel_err(da[0, r], ref_da[0, 0]) <= TOL32, r
        assert rel_err(dx[0, r], ref_dx[0, 0]) <= TOL32, r
        assert rel_err(dh0[:, r], ref_dh0[:, 0]) <= TOL32, r
    del h, da, dx, dh0, w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("variant", ["planner", "stream"])
def test_full_packed_bidir_all_channels(lib, variant):
    """Every output of the packed bidirectional workload (2048 channels, 64
    sequences, bf16 inputs, both branches) against the oracle, channel batch
    by channel batch: h and dh0 (fp32) within 1e-5, da and dx (stored in
    bf16) within 1e-2."""
    w = workloads.packed_bidir(seed=0)
    g = cuda(w.af, w.xf, w.ar, w.xr, w.cu_seqlens, w.dhf, w.dhr)
    af, xf, ar, xr, cu, dhf, dhr = g
    opts = {"variant": lib.SCAN_VARIANT_STREAM} if variant == "stream" else None
    hf, hr = lib.scan_bidir_fwd(af, xf, ar, xr, None, None, cu, opts=opts)
    daf, dxf, dh0f, dar, dxr, dh0r = lib.scan_bidir_bwd(af, hf, dhf, ar, hr, dhr, None, None, cu,
                                                        opts=opts)
    torch.cuda.synchronize()
    assert lib.scan_get_device_status(DEV) == lib.SCAN_OK
    del af, xf, ar, xr, dhf, dhr
    dh0f, dh0r = dh0f.cpu(), dh0r.cpu()
    branches = ((w.af, w.xf, w.dhf, hf, daf, dxf, dh0f, False),
                (w.ar, w.xr, w.dhr, hr, dar, dxr, dh0r, True))

    def check(c0, c1):
        e = {}
        for (a, x, dh, h, da, dx, dh0, rev) in branches:
            ra, rx, rdh = a[c0:c1], x[c0:c1], dh[c0:c1]
            ref_h = oracle.scan_fwd(ra, rx, None, w.cu_seqlens, rev)
            ref_da, ref_dx, ref_dh0 = oracle.scan_bwd(ra, rx, rdh, None, w.cu_seqlens, rev)
            tag = "r" if rev else "f"
            e["h" + tag] = max_rel(h[c0:c1], ref_h)
            e["da" + tag] = max_rel(da[c0:c1], ref_da)
            e["dx" + tag] = max_rel(dx[c0:c1], ref_dx)
            e["dh0" + tag] = max_rel(dh0[:, c0:c1], ref_dh0)
        return e

    errs = sweep(w.af.shape[0], 32, check)
    print("packed_bidir all channels", variant, errs)
    assert errs["items"] == 2048
    assert all(errs[k] <= TOL32 for k in ("hf", "hr", "dh0f", "dh0r")), errs
    assert all(errs[k] <= TOLBF for k in ("daf", "dar", "dxf", "dxr")), errs


def test_full_log_4k_all_rows(lib):
    """Every output of the log-space workload (8 x 1536 x 4096), forward and
    backward, against the oracle."""
    w = workloads.log_4k(seed=0)
    B, C, T = w.log_a.shape
    ga, gx = cuda(w.log_a, w.log_x)
    h = lib.scan_log_fwd(ga, gx)
    dla, dlx, dlh0 = lib.scan_log_bwd(ga, gx, h, w.dh.to(DEV))
    torch.cuda.synchronize()
    assert lib.scan_get_device_status(DEV) == lib.SCAN_OK
    la, lx, dh2 = (t.view(B * C, T) for t in (w.log_a, w.log_x, w.dh))
    h2, dla2, dlx2 = (t.view(B * C, T) for t in (h, dla, dlx))
    dlh0f = dlh0.view(-1).cpu()

    def check(r0, r1):
        ra, rx, rdh = la[r0:r1][None], lx[r0:r1][None], dh2[r0:r1][None]
        ref = oracle.scan_log_fwd(ra, rx)
        rg = oracle.scan_log_bwd(ra, rx, rdh)
        return {"h": max_rel(h2[r0:r1], ref[0]), "dlog_a": max_rel(dla2[r0:r1], rg[0][0]),
                "dlog_x": max_rel(dlx2[r0:r1], rg[1][0]),
                "dlog_h0": max_rel(dlh0f[r0:r1], rg[2][0])}

    errs = sweep(B * C, 512, check)
    print("log_4k all rows", errs)
    assert errs["items"] == B * C
    assert all(errs[k] <= TOL32 for k in ("h", "dlog_a", "dlog_x", "dlog_h0")), errs
