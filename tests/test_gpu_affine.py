"""GPU parity of the block-matrix affine scan against the fp64 oracle.

H_t = A_t H_{t-1} + B_t and its backward ("Triton scan kernels": One
associative-scan family; Autograd integration and the reversed-scan backward),
through the C ABI. The products do not commute, so any order mistake shows up
against the oracle.

Tolerance, fp32: max |got - ref| / max(1, |ref|) <= 1e-5 for H and dB. dA_t =
G_t H_{t-1}^T and dh0 = A_0^T G_0 are k-term contractions of those fp32
results, so their error is bounded by the magnitudes of their terms, not by
the result (cancellation): if G and H each meet e in the max(1, |.|) metric,
dA_il is within 2e sum_j max(1, |G_ij|) max(1, |H_lj|). Their error is
normalised by that term scale (resp. sum_l |A_li| max(1, |G_lj|) for dh0),
computed from the oracle's own values. Beside that gate, the plain metric
max |got - ref| / max(1, |ref|) of dA and dh0 is computed, printed and held to
1e-3, the gate "Triton scan kernels" (Conformance) puts on affine gradients.
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from _sweep import max_rel, sweep, worst
from associative_affine_scan_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = 1e-5
TOL_GRAD_PLAIN = 1e-3
DEV = torch.device("cuda", 0)
HERE = os.path.dirname(os.path.abspath(__file__))


def rel_err(got, ref, scale=None):
    got = got.detach().double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    ref = np.asarray(ref, dtype=np.float64)
    den = np.maximum(1.0, np.abs(ref))
    if scale is not None:
        den = np.maximum(den, scale)
    return 0.0 if got.size == 0 else float(np.max(np.abs(got - ref) / den))


def contraction_scales(A, h0, ref_H, ref_dB):
    """Term scales of the dA and dh0 contractions (see the module docstring)."""
    A = np.asarray(A.double() if isinstance(A, torch.Tensor) else A, dtype=np.float64)
    G = np.maximum(1.0, np.abs(ref_dB))
    prev = np.empty_like(ref_H)
    prev[:, 1:] = ref_H[:, :-1]
    prev[:, 0] = 0.0 if h0 is None else np.asarray(h0.double())
    dA_scale = np.einsum("btnij,btnlj->btnil", G, np.maximum(1.0, np.abs(prev)))
    dh0_scale = np.einsum("bnli,bnlj->bnij", np.abs(A[:, 0]), G[:, 0])
    return dA_scale, dh0_scale


def run_and_check(lib, w, opts=None):
    A, Bm, dH = w.A.to(DEV), w.Bm.to(DEV), w.dH.to(DEV)
    h0 = w.h0.to(DEV) if w.h0 is not None else None
    H = lib.affine_scan_fwd(A, Bm, h0, opts=opts)
    dA, dB, dh0 = lib.affine_scan_bwd(A, H, dH, h0, opts=opts)
    torch.cuda.synchronize()
    assert lib.scan_get_device_status(DEV) == lib.SCAN_OK
    ref_H = oracle.affine_fwd(w.A, w.Bm, w.h0)
    ref_dA, ref_dB, ref_dh0 = oracle.affine_bwd(w.A, w.Bm, w.dH, w.h0)
    sA, s0 = contraction_scales(w.A, w.h0, ref_H, ref_dB)
    errs = {"H": rel_err(H, ref_H), "dA": rel_err(dA, ref_dA, sA), "dB": rel_err(dB, ref_dB),
            "dh0": rel_err(dh0, ref_dh0, s0)}
    plain = {"dA": rel_err(dA, ref_dA), "dh0": rel_err(dh0, ref_dh0)}
    print("affine", tuple(w.A.shape), "plain-metric gradient error", plain)
    assert all(v <= TOL for v in errs.values()), errs
    assert all(v <= TOL_GRAD_PLAIN for v in plain.values()), plain
    return plain


AFFINE_VARIANTS = {"planner": None, "stationary": {"variant": 1}, "lookback": {"variant": 2}}


@pytest.mark.parametrize("T", [1, 5, 15, 16, 17, 63, 64, 65, 200, 1000])
@pytest.mark.parametrize("N", [1, 7, 8, 9, 37, 70])
@pytest.mark.parametrize("variant", list(AFFINE_VARIANTS))
def test_affine_4x4_shapes(lib, T, N, variant):
    """4 x 4 blocks under the planner and each variant: STATIONARY runs the
    ring kernel where it applies (N >= 8, T >= 16: one warp per 8 lanes,
    stage edges at 16-step multiples) and the look-back kernel elsewhere."""
    for h0 in (True, False):
        w = workloads.affine(2, T, N, 4, 4, seed=T * 100 + N, h0=h0)
        run_and_check(lib, w, AFFINE_VARIANTS[variant])


def test_affine_4x4_stationary_many_groups(lib):
    """The ring kernel with several lane groups per batch row, a partial last
    group (N = 203) and a ragged last stage (T = 1001)."""
    w = workloads.affine(3, 1001, 203, 4, 4, seed=5, h0=True)
    run_and_check(lib, w, {"variant": 1})


@pytest.mark.parametrize("chunk", [64, 128, 256])
def test_affine_chunk_sizes(lib, chunk):
    w = workloads.affine(1, 777, 33, 4, 4, seed=chunk, h0=True)
    run_and_check(lib, w, {"chunk": chunk})


def test_affine_2x2(lib):
    w = workloads.affine(3, 513, 40, 2, 2, seed=5, h0=True)
    run_and_check(lib, w)


ENVELOPE = [(k, v) for k in (1, 2, 4, 8, 16) for v in (1, 2, 4, 8, 16)]


@pytest.mark.parametrize("k,v", ENVELOPE)
def test_affine_envelope(lib, k, v):
    """Every block shape of the envelope, forward and backward, over several
    chunks (T = 131 at 64-step chunks) and a partial group of lanes (N = 5)."""
    w = workloads.affine(2, 131, 5, k, v, seed=17 * k + v, h0=True)
    run_and_check(lib, w)


@pytest.mark.parametrize("k,v", [(1, 16), (16, 1), (8, 2)])
def test_affine_envelope_longer_chunks_and_no_h0(lib, k, v):
    w = workloads.affine(1, 700, 9, k, v, seed=k + 100 * v, h0=False)
    run_and_check(lib, w, {"chunk": 256})


def test_affine_k1_is_the_scalar_scan(lib):
    """k = v = 1 is h_t = a_t h_{t-1} + x_t: the same values as the scalar
    forward on the same inputs (one lane per channel)."""
    B, T, N = 2, 300, 7
    g = torch.Generator().manual_seed(3)
    a = torch.rand((B, T, N), generator=g)
    x = torch.randn((B, T, N), generator=g)
    H = lib.affine_scan_fwd(a.view(B, T, N, 1, 1).to(DEV), x.view(B, T, N, 1, 1).to(DEV))
    h = lib.scan_fwd(a.permute(0, 2, 1).contiguous().to(DEV), x.permute(0, 2, 1).contiguous().to(DEV))
    torch.cuda.synchronize()
    ref = oracle.scan_fwd(a.permute(0, 2, 1).contiguous(), x.permute(0, 2, 1).contiguous())
    assert rel_err(H.view(B, T, N).permute(0, 2, 1), ref) <= TOL
    assert rel_err(h, ref) <= TOL


def prefix_reference(A, dAbar):
    """The coefficient prefix is the block scan with v = k, B = 0, h0 = I."""
    B, T, N, k, _ = A.shape
    zeros = torch.zeros_like(A)
    eye = torch.eye(k).expand(B, N, k, k).contiguous()
    ref = oracle.affine_fwd(A, zeros, eye)
    ref_dA = oracle.affine_bwd(A, zeros, dAbar, eye)[0]
    # term scale of dA_t = G_t Abar_{t-1}^T (module docstring)
    G = np.maximum(1.0, np.abs(oracle.affine_bwd(A, zeros, dAbar, eye)[1]))
    prev = np.empty_like(ref)
    prev[:, 1:] = ref[:, :-1]
    prev[:, 0] = np.asarray(eye.double())
    scale = np.einsum("btnij,btnlj->btnil", G, np.maximum(1.0, np.abs(prev)))
    return ref, ref_dA, scale


@pytest.mark.parametrize("k", [1, 2, 4, 8, 16])
def test_affine_prefix(lib, k):
    w = workloads.affine(2, 150, 5, k, k, seed=31 + k)
    dAbar = w.dH
    Abar = lib.affine_prefix_fwd(w.A.to(DEV))
    dA = lib.affine_prefix_bwd(w.A.to(DEV), Abar, dAbar.to(DEV))
    torch.cuda.synchronize()
    assert lib.scan_get_device_status(DEV) == lib.SCAN_OK
    ref, ref_dA, scale = prefix_reference(w.A, dAbar)
    assert rel_err(Abar, ref) <= TOL
    assert rel_err(dA, ref_dA, scale) <= TOL


def test_affine_prefix_gradient_accumulates(lib):
    """accumulate=True adds the prefix's dA term to the state's dA. (The two
    prefix backward runs compared here may differ by rounding: the look-back
    composes whichever earlier records are already published.)"""
    w = workloads.affine(1, 200, 9, 4, 4, seed=77, h0=True)
    A, Bm, dH, h0 = w.A.to(DEV), w.Bm.to(DEV), w.dH.to(DEV), w.h0.to(DEV)
    H = lib.affine_scan_fwd(A, Bm, h0)
    dA_state, _, _ = lib.affine_scan_bwd(A, H, dH, h0)
    Abar = lib.affine_prefix_fwd(A)
    dAbar = torch.randn(A.shape, generator=torch.Generator().manual_seed(5)).to(DEV)
    dA_prefix = lib.affine_prefix_bwd(A, Abar, dAbar)
    both = lib.affine_prefix_bwd(A, Abar, dAbar, dA_state.clone(), accumulate=True)
    torch.cuda.synchronize()
    assert rel_err(both, (dA_state + dA_prefix).double().cpu().numpy()) <= TOL


def test_affine_golden_worked_example_bit_exact(lib):
    with open(os.path.join(HERE, "golden", "affine_2x2_dyadic.json")) as f:
        g = json.load(f)
    A, Bm, h0, dH = (torch.tensor(g[k], dtype=torch.float32, device=DEV)
                     for k in ("A", "Bm", "h0", "dH"))
    H = lib.affine_scan_fwd(A, Bm, h0)
    dA, dB, dh0 = lib.affine_scan_bwd(A, H, dH, h0)
    assert H.cpu().tolist() == g["H"]
    assert dB.cpu().tolist() == g["dB"]
    assert dA.cpu().tolist() == g["dA"]
    assert dh0.cpu().tolist() == g["dh0"]


def test_affine_identity_is_cumsum_exactly(lib):
    T, N = 300, 32
    A = torch.eye(4).expand(1, T, N, 4, 4).contiguous().to(DEV)
    Bm = torch.randint(-3, 4, (1, T, N, 4, 4)).float().to(DEV)
    H = lib.affine_scan_fwd(A, Bm)
    assert torch.equal(H, torch.cumsum(Bm, dim=1))


def test_affine_rejects_unsupported_and_misaligned(lib):
    A = torch.zeros(1, 4, 2, 3, 3, device=DEV)
    Bm = torch.zeros(1, 4, 2, 3, 3, device=DEV)
    with pytest.raises(lib.ScanError) as e:
        lib.affine_scan_fwd(A, Bm)
    assert e.value.status == lib.SCAN_ERR_UNSUPPORTED
    buf = torch.zeros(1 + 2 * 4 * 16, device=DEV)
    A = buf[1:].view(1, 4, 2, 4, 4)
    with pytest.raises(lib.ScanError) as e:
        lib.affine_scan_fwd(A, torch.zeros(1, 4, 2, 4, 4, device=DEV))
    assert e.value.status == lib.SCAN_ERR_ALIGNMENT


def test_affine_ring_wait_limit_reports_timeout(lib):
    """The ring kernel's first warp waits at its second stage on an mbarrier
    that nothing completes: the wait expires after 1 ms, the status reads
    SCAN_ERR_TIMEOUT, and the next call runs normally."""
    w = workloads.affine(1, 600, 32, 4, 4, seed=19, h0=True)
    A, Bm, h0, dH = w.A.to(DEV), w.Bm.to(DEV), w.h0.to(DEV), w.dH.to(DEV)
    lib.scan_get_device_status(DEV)
    opts = {"variant": lib.SCAN_VARIANT_STATIONARY, "test_stall": 1, "wait_limit_s": 1e-3}
    H = lib.affine_scan_fwd(A, Bm, h0, opts=opts)
    assert lib.scan_get_device_status(DEV) == lib.SCAN_ERR_TIMEOUT
    lib.affine_scan_bwd(A, H, dH, h0, opts=opts)
    assert lib.scan_get_device_status(DEV) == lib.SCAN_ERR_TIMEOUT
    H = lib.affine_scan_fwd(A, Bm, h0, opts={"variant": lib.SCAN_VARIANT_STATIONARY})
    assert lib.scan_get_device_status(DEV) == lib.SCAN_OK
    assert rel_err(H, oracle.affine_fwd(w.A, w.Bm, w.h0)) <= TOL


def test_affine_wait_limit_reports_timeout(lib):
    w = workloads.affine(1, 600, 32, 4, 4, seed=9, h0=True)
    A, Bm, h0 = w.A.to(DEV), w.Bm.to(DEV), w.h0.to(DEV)
    lib.scan_get_device_status(DEV)
    lib.affine_scan_fwd(A, Bm, h0, opts={"chunk": 128, "test_stall": 1, "wait_limit_s": 1e-3})
    assert lib.scan_get_device_status(DEV) == lib.SCAN_ERR_TIMEOUT
    H = lib.affine_scan_fwd(A, Bm, h0, opts={"chunk": 128})
    assert lib.scan_get_device_status(DEV) == lib.SCAN_OK
    assert rel_err(H, oracle.affine_fwd(w.A, w.Bm, w.h0)) <= TOL


def test_full_affine_4x4_all_lanes(lib):
    """Every output of the 8 x 4096 x 256 block workload (k = v = 4) against the
    oracle, in batches of 32 lanes: H and dB within 1e-5 of max(1, |ref|), dA
    and dh0 within 1e-5 of their term scale and within 1e-3 in the plain
    metric (both printed)."""
    w = workloads.affine_4x4(seed=0)
    A, Bm, dH = w.A.to(DEV), w.Bm.to(DEV), w.dH.to(DEV)
    H = lib.affine_scan_fwd(A, Bm)
    dA, dB, dh0 = lib.affine_scan_bwd(A, H, dH)
    torch.cuda.synchronize()
    assert lib.scan_get_device_status(DEV) == lib.SCAN_OK
    del A, Bm, dH
    B, T, N = w.A.shape[:3]
    lanes = 32
    groups = (N + lanes - 1) // lanes

    def check(i0, i1):
        e = {}
        for i in range(i0, i1):
            b, n0 = i // groups, (i % groups) * lanes
            sl = (slice(b, b + 1), slice(None), slice(n0, min(N, n0 + lanes)))
            ref_H = oracle.affine_fwd(w.A[sl], w.Bm[sl])
            ref_dA, ref_dB, ref_dh0 = oracle.affine_bwd(w.A[sl], w.Bm[sl], w.dH[sl])
            sA, s0 = contraction_scales(w.A[sl], None, ref_H, ref_dB)
            got_dh0 = dh0[b:b + 1, sl[2]]
            for k, v in (("H", max_rel(H[sl], ref_H)), ("dB", max_rel(dB[sl], ref_dB)),
                         ("dA", max_rel(dA[sl], ref_dA, sA)), ("dh0", max_rel(got_dh0, ref_dh0, s0)),
                         ("dA_plain", max_rel(dA[sl], ref_dA)),
                         ("dh0_plain", max_rel(got_dh0, ref_dh0))):
                e[k] = worst(e.get(k, 0.0), v)
        return e

    errs = sweep(B * groups, 1, check)
    print("affine_4x4 all lanes", errs)
    assert errs["items"] == B * groups
    assert all(errs[k] <= TOL for k in ("H", "dB", "dA", "dh0")), errs
    assert errs["dA_plain"] <= TOL_GRAD_PLAIN and errs["dh0_plain"] <= TOL_GRAD_PLAIN, errs
