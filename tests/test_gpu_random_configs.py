"""Seeded random configurations of every entry point against the fp64 oracle.

The per-feature tests enumerate each option on its own; here each case draws
all of them at once (seeded, so every run checks the same cases): dtype,
dense or packed rows, direction, initial state, resets, the carry scheme,
chunk length, rows per block, stationary segments and stream stages for the
scalar scan and its two-branch and log-space forms; block shapes from the
whole (k, v) envelope with each scheme; GDN state shapes and lengths; RG-LRU
sizes and document mixes. Tolerances are those of the per-feature tests.
"""

import numpy as np
import pytest
import torch

import oracle
from test_gpu_affine import run_and_check
from test_gpu_gdn import check as gdn_check
from test_gpu_rglru import compare as rglru_compare, run as rglru_run, within as rglru_within
from test_gpu_scalar import TOL32, TOLBF, check_fwd_bwd, cuda, rel_err
from associative_affine_scan_gb300 import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def draw_T(rng, hi=3000):
    """Lengths biased to the chunk edges (multiples of 128 +- 1) and tiny rows."""
    kind = rng.integers(0, 3)
    if kind == 0:
        return int(rng.integers(1, 9))
    if kind == 1:
        return max(1, int(128 * rng.integers(1, hi // 128 + 1) + rng.integers(-1, 2)))
    return int(rng.integers(1, hi + 1))


def draw_opts(rng, lib):
    variant = int(rng.choice([lib.SCAN_VARIANT_AUTO, lib.SCAN_VARIANT_STATIONARY,
                              lib.SCAN_VARIANT_LOOKBACK, lib.SCAN_VARIANT_STREAM]))
    opts = {"variant": variant}
    if rng.random() < 0.6:
        opts["chunk"] = int(rng.choice([128, 256, 512]))
    if rng.random() < 0.5:
        opts["rows_per_cta"] = int(rng.integers(1, 9))
    if variant == lib.SCAN_VARIANT_STATIONARY and rng.random() < 0.5:
        opts["segments"] = int(rng.integers(1, 6))
    if variant == lib.SCAN_VARIANT_STREAM and rng.random() < 0.5:
        opts["stages"] = int(rng.choice([2, 3, 4, 8]))
    return opts


def packed_lengths(rng):
    n = int(rng.integers(1, 13))
    lens = rng.integers(0, 700, size=n)
    lens[rng.random(n) < 0.15] = 0  # empty sequences
    if lens.sum() == 0:
        lens[0] = 1
    cu = np.zeros(n + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    return torch.from_numpy(cu)


def scalar_inputs(rng, seed, shape, dtype, n_h0_rows=None):
    g = torch.Generator().manual_seed(seed)
    a = torch.rand(shape, generator=g)
    a[torch.rand(shape, generator=g) < 0.01] = 0.0  # resets
    x = torch.randn(shape, generator=g)
    dh = torch.randn(shape, generator=g)
    h0 = None
    if rng.random() < 0.5:
        h0 = torch.randn(n_h0_rows if n_h0_rows is not None else shape[:2], generator=g)
    return a.to(dtype), x.to(dtype), dh, h0


@pytest.mark.parametrize("i", range(120))
def test_random_scalar(lib, i):
    rng = np.random.default_rng(7000 + i)
    dtype = torch.bfloat16 if rng.random() < 0.4 else torch.float32
    reverse = bool(rng.random() < 0.5)
    opts = draw_opts(rng, lib)
    if rng.random() < 0.4:
        cu = packed_lengths(rng)
        C = int(rng.integers(1, 25))
        a, x, dh, h0 = scalar_inputs(rng, 7000 + i, (C, int(cu[-1])), dtype,
                                     (cu.numel() - 1, C))
    else:
        cu = None
        shape = (int(rng.integers(1, 4)), int(rng.integers(1, 21)), draw_T(rng))
        a, x, dh, h0 = scalar_inputs(rng, 7000 + i, shape, dtype)
    check_fwd_bwd(lib, a, x, dh, h0, cu, reverse, opts=opts)


@pytest.mark.parametrize("i", range(30))
def test_random_bidir(lib, i):
    rng = np.random.default_rng(8000 + i)
    dtype = torch.bfloat16 if rng.random() < 0.5 else torch.float32
    opts = draw_opts(rng, lib)
    cu = packed_lengths(rng)
    C = int(rng.integers(1, 17))
    T = int(cu[-1])
    af, xf, dhf, h0f = scalar_inputs(rng, 8000 + i, (C, T), dtype, (cu.numel() - 1, C))
    ar, xr, dhr, h0r = scalar_inputs(rng, 8500 + i, (C, T), dtype, (cu.numel() - 1, C))
    if (h0f is None) != (h0r is None):
        h0r = None if h0f is None else torch.randn_like(h0f)
    g = cuda(af, xf, ar, xr, dhf, dhr, h0f, h0r, cu)
    hf, hr = lib.scan_bidir_fwd(g[0], g[1], g[2], g[3], g[6], g[7], g[8], opts=opts)
    grads = lib.scan_bidir_bwd(g[0], hf, g[4], g[2], hr, g[5], g[6], g[7], g[8], opts=opts)
    torch.cuda.synchronize()
    assert lib.scan_get_device_status(DEV) == lib.SCAN_OK
    tol_g = TOLBF if dtype == torch.bfloat16 else TOL32
    ref_f = oracle.scan_bwd(af, xf, dhf, h0f, cu, False)
    ref_r = oracle.scan_bwd(ar, xr, dhr, h0r, cu, True)
    assert rel_err(hf, oracle.scan_fwd(af, xf, h0f, cu, False)) <= TOL32
    assert rel_err(hr, oracle.scan_fwd(ar, xr, h0r, cu, True)) <= TOL32
    daf, dxf, dh0f, dar, dxr, dh0r = grads
    for got, ref, tol in ((daf, ref_f[0], tol_g), (dxf, ref_f[1], tol_g), (dh0f, ref_f[2], TOL32),
                          (dar, ref_r[0], tol_g), (dxr, ref_r[1], tol_g), (dh0r, ref_r[2], TOL32)):
        assert rel_err(got, ref) <= tol


@pytest.mark.parametrize("i", range(30))
def test_random_log(lib, i):
    rng = np.random.default_rng(9000 + i)
    reverse = bool(rng.random() < 0.5)
    opts = draw_opts(rng, lib)
    g = torch.Generator().manual_seed(9000 + i)
    if rng.random() < 0.4:
        cu = packed_lengths(rng)
        shape = (int(rng.integers(1, 17)), int(cu[-1]))
        h0_shape = (cu.numel() - 1, shape[0])
    else:
        cu = None
        shape = (int(rng.integers(1, 4)), int(rng.integers(1, 17)), draw_T(rng))
        h0_shape = shape[:2]
    la = torch.nn.functional.logsigmoid(torch.randn(shape, generator=g))
    la[torch.rand(shape, generator=g) < 0.01] = -float("inf")
    lx = torch.randn(shape, generator=g)
    dh = torch.randn(shape, generator=g)
    lh0 = torch.randn(h0_shape, generator=g) if rng.random() < 0.5 else None
    ga, gx, gdh, gh0, gcu = cuda(la, lx, dh, lh0, cu)
    h = lib.scan_log_fwd(ga, gx, gh0, gcu, reverse, opts=opts)
    dla, dlx, dlh0 = lib.scan_log_bwd(ga, gx, h, gdh, gh0, gcu, reverse, opts=opts)
    torch.cuda.synchronize()
    assert lib.scan_get_device_status(DEV) == lib.SCAN_OK
    assert rel_err(h, oracle.scan_log_fwd(la, lx, lh0, cu, reverse)) <= TOL32
    ref = oracle.scan_log_bwd(la, lx, dh, lh0, cu, reverse)
    assert rel_err(dla, ref[0]) <= TOL32 and rel_err(dlx, ref[1]) <= TOL32
    if lh0 is not None:
        assert rel_err(dlh0, ref[2]) <= TOL32


@pytest.mark.parametrize("i", range(30))
def test_random_affine(lib, i):
    rng = np.random.default_rng(10000 + i)
    k, v = (int(rng.choice([1, 2, 4, 8, 16])) for _ in range(2))
    B, N = int(rng.integers(1, 4)), int(rng.integers(1, 13))
    T = int(rng.integers(1, 600 if k * v <= 16 else 200))
    w = workloads.affine(B, T, N, k, v, seed=10000 + i, h0=bool(rng.random() < 0.5))
    opts = [None, {"variant": 1}, {"variant": 2}][int(rng.integers(0, 3))]
    run_and_check(lib, w, opts)


@pytest.mark.parametrize("i", range(16))
def test_random_gdn(lib, i):
    rng = np.random.default_rng(11000 + i)
    S, D = (int(rng.choice([16, 32])) for _ in range(2))
    w = workloads.gdn(int(rng.integers(1, 3)), int(rng.integers(1, 6)), draw_T(rng, 400), S, D,
                      seed=11000 + i, h0=bool(rng.random() < 0.5))
    zero = torch.rand(w.alpha.shape, generator=torch.Generator().manual_seed(i)) < 0.02
    w.alpha[zero] = 0.0
    gdn_check(lib, w)


@pytest.mark.parametrize("i", range(16))
def test_random_rglru(lib, i):
    rng = np.random.default_rng(12000 + i)
    docs = [None, (1, 40), (100, 600)][int(rng.integers(0, 3))]
    dtype = torch.bfloat16 if rng.random() < 0.4 else torch.float32
    w = workloads.rglru(int(rng.integers(1, 11)), int(rng.integers(1, 9)), draw_T(rng, 1500),
                        seed=12000 + i, docs=docs, h0=bool(rng.random() < 0.5), dtype=dtype)
    h, g = rglru_run(lib, w, shift=int(rng.integers(0, 2)))
    errs = rglru_compare(w, h, g)
    assert rglru_within(errs, dtype), errs
