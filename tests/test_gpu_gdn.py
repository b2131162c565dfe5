"""GPU parity of the scalar-gated outer-product state against the fp64 oracle.

h_t = alpha_t h_{t-1} + b_t v_t^T, o_t = h_t^T c_t per (batch, head), and the
reverse-time backward ("Operations & Triton Kernels" (HyMo): The chunked GDN
algorithm; Mathematical Derivation of the Reverse-Time Backward Pass), through
the C ABI.

Tolerance, fp32: o, dv, db, dc and dh0 are sums over S or D products of fp32
values, dalpha a sum over S * D; each error is normalised by the sum of the
absolute values of its terms, which the oracle computes by running on
|alpha|, |b|, |v|, |c|, |h0|, |dout| (every term becomes its absolute value),
and must stay within 1e-5 of it (or of max(1, |ref|), whichever is larger).
The plain metric max |got - ref| / max(1, |ref|) of every gradient is
computed beside it, printed, and held to 1e-3 (the gate "Triton scan kernels",
Conformance, puts on gradients of the affine scan).
"""

import numpy as np
import pytest
import torch

import oracle
from _sweep import sweep, worst
from associative_affine_scan_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = 1e-5
TOL_GRAD_PLAIN = 1e-3
DEV = torch.device("cuda", 0)


def err(got, ref, scale=None):
    got = got.detach().double().cpu().numpy()
    den = np.maximum(1.0, np.abs(ref))
    if scale is not None:
        den = np.maximum(den, scale)
    return 0.0 if got.size == 0 else float(np.max(np.abs(got - ref) / den))


GRADS = ("dalpha", "db", "dv", "dc", "dh0")


def check(lib, w, plain_gate=True):
    alpha, b, v, c, dout = (t.to(DEV) for t in (w.alpha, w.b, w.v, w.c, w.dout))
    h0 = w.h0.to(DEV) if w.h0 is not None else None
    o, ck = lib.gdn_fwd(alpha, b, v, c, h0)
    g = lib.gdn_bwd(alpha, b, v, c, ck, dout)
    torch.cuda.synchronize()
    ref_o = oracle.gdn_fwd(w.alpha, w.b, w.v, w.c, w.h0)
    ref_g = oracle.gdn_bwd(w.alpha, w.b, w.v, w.c, w.dout, w.h0)
    ab = lambda t: None if t is None else t.abs()
    sc_o = oracle.gdn_fwd(ab(w.alpha), ab(w.b), ab(w.v), ab(w.c), ab(w.h0))
    sc_g = oracle.gdn_bwd(ab(w.alpha), ab(w.b), ab(w.v), ab(w.c), ab(w.dout), ab(w.h0))
    errs = {"o": err(o, ref_o, sc_o)}
    plain = {"o": err(o, ref_o)}
    for name, got, ref, sc in zip(GRADS, g, ref_g, sc_g):
        errs[name] = err(got, ref, sc)
        plain[name] = err(got, ref)
    print("gdn", tuple(w.b.shape), "term-scale error", errs, "plain-metric error", plain)
    assert all(v <= TOL for v in errs.values()), errs
    if plain_gate:
        assert all(plain[k] <= TOL_GRAD_PLAIN for k in GRADS), plain


# T covers the backward's 32-step chunks (31, 32, 33), the forward's 64-step
# chunks (63, 64, 65) and the checkpoint a forward chunk writes in its middle
# (96, 97), with ragged tails.
@pytest.mark.parametrize("S,D", [(16, 16), (16, 32), (32, 16), (32, 32)])
@pytest.mark.parametrize("T", [1, 5, 16, 17, 31, 32, 33, 63, 64, 65, 96, 97, 130, 257])
def test_gdn_shapes(lib, S, D, T):
    for h0 in (True, False):
        w = workloads.gdn(2, 3, T, S, D, seed=T * 7 + S + D + h0, h0=h0)
        check(lib, w)


@pytest.mark.parametrize("S,D", [(16, 16), (16, 32), (32, 16), (32, 32)])
@pytest.mark.parametrize("T", [1, 15, 16, 17, 31, 32, 33, 100])
def test_gdn_many_heads(lib, S, D, T):
    """160 heads (more than one per SM) at ragged T around the 16- and 32-step
    edges, with and without h0."""
    for h0 in (True, False):
        w = workloads.gdn(8, 20, T, S, D, seed=T * 13 + S + D + h0, h0=h0)
        check(lib, w)


def test_gdn_with_one_by_one_state_matches_the_scalar_scan(lib):
    """Identity through the reduction: with b_t = e_0, c_t = e_0 and v_t = x_t e_0,
    o_t[0] is the scalar scan h_t = alpha_t h_{t-1} + x_t."""
    B, H, T, S, D = 1, 4, 300, 16, 16
    g = torch.Generator().manual_seed(8)
    alpha = torch.rand((B, H, T), generator=g)
    x = torch.randn((B, H, T), generator=g)
    b = torch.zeros(B, H, T, S)
    b[..., 0] = 1.0
    c = b.clone()
    v = torch.zeros(B, H, T, D)
    v[..., 0] = x
    o, _ = lib.gdn_fwd(alpha.to(DEV), b.to(DEV), v.to(DEV), c.to(DEV), checkpoints=False)
    torch.cuda.synchronize()
    ref = oracle.scan_fwd(alpha.view(1, B * H, T), x.view(1, B * H, T))
    assert np.allclose(o[..., 0].cpu().double().numpy().reshape(1, B * H, T), ref,
                       rtol=1e-5, atol=1e-6)


def test_gdn_rejects_unsupported_shapes(lib):
    a = torch.rand(1, 1, 8, device=DEV)
    b = torch.zeros(1, 1, 8, 8, device=DEV)
    with pytest.raises(lib.ScanError) as e:
        lib.gdn_fwd(a, b, b, b)
    assert e.value.status == lib.SCAN_ERR_UNSUPPORTED


def test_gdn_4k_all_heads(lib):
    """Every output of the bench workload (8 x 32 heads x 4096 steps, 32 x 32
    state) against the oracle, head by head on the host cores: within 1e-5 of
    the term scale, and the gradients within 1e-3 in the plain metric."""
    w = workloads.gdn_4k(seed=0)
    alpha, b, v, c, dout = (t.to(DEV) for t in (w.alpha, w.b, w.v, w.c, w.dout))
    o, ck = lib.gdn_fwd(alpha, b, v, c)
    outs = lib.gdn_bwd(alpha, b, v, c, ck, dout)
    torch.cuda.synchronize()
    assert lib.scan_get_device_status(DEV) == lib.SCAN_OK
    B, H = w.alpha.shape[:2]

    def check(i0, i1):
        e = {}
        for i in range(i0, i1):
            bb, hh = divmod(i, H)
            sl = lambda t: t[bb:bb + 1, hh:hh + 1]
            ins = [sl(t) for t in (w.alpha, w.b, w.v, w.c)]
            ref_o = oracle.gdn_fwd(*ins)
            ref_g = oracle.gdn_bwd(*ins, sl(w.dout))
            absin = [t.abs() for t in ins]
            sc_o = oracle.gdn_fwd(*absin)
            sc_g = oracle.gdn_bwd(*absin, sl(w.dout).abs())
            vals = [("o", err(sl(o), ref_o, sc_o))]
            for name, got, ref, sc in zip(GRADS, outs, ref_g, sc_g):
                vals.append((name, err(sl(got), ref, sc)))
                vals.append((name + "_plain", err(sl(got), ref)))
            for k, val in vals:
                e[k] = worst(e.get(k, 0.0), val)
        return e

    errs = sweep(B * H, 4, check)
    print("gdn_4k all heads", errs)
    assert errs["items"] == B * H
    assert all(errs[k] <= TOL for k in ("o",) + GRADS), errs
    assert all(errs[k + "_plain"] <= TOL_GRAD_PLAIN for k in GRADS), errs


@pytest.mark.parametrize("T", [64, 200])
def test_gdn_gate_zero_resets(lib, T):
    """alpha_t = 0 erases the state (h_t = b_t v_t^T). Zero gates at a chunk's
    first and last steps and inside it; the backward's per-chunk gate
    products are formed without division, so dalpha stays exact there."""
    w = workloads.gdn(2, 2, T, 32, 32, seed=11 + T, h0=True)
    for t in (0, 1, 31, 32, 63, 64, 95, 96, 127, 128, 199):
        if t < T:
            w.alpha[:, :, t] = 0.0
    w.alpha[1, 1, :] = 0.0  # every step a reset
    check(lib, w)


@pytest.mark.parametrize("S,D", [(32, 32), (32, 16), (16, 16)])
@pytest.mark.parametrize("T", [64, 130, 257])
def test_gdn_gate_regimes(lib, S, D, T):
    """Heads whose gates leave the forward walk's frame range within a chunk
    and restart it: gates in (0, 0.2) (the product falls below 2^-20 every
    few steps), gates in (1.1, 1.4) (it rises above 2^20), gates of 1e-8 and 0
    between ordinary ones, and ordinary gates near 1. Gates above 1 grow the
    state and its adjoint by up to 1e25 over the sequence, and gradient
    entries far below their terms come out of cancellation: there the
    term-scale metric is the gate (the plain metric is printed only)."""
    w = workloads.gdn(2, 4, T, S, D, seed=5 * T + S + D, h0=True)
    g = torch.Generator().manual_seed(T + 7)
    shape = (2, T)
    w.alpha[:, 0] = 0.2 * torch.rand(shape, generator=g)
    w.alpha[:, 1] = 1.1 + 0.3 * torch.rand(shape, generator=g)
    mixed = torch.sigmoid(torch.randn(shape, generator=g) + 3.0)
    pick = torch.rand(shape, generator=g)
    mixed[pick < 0.1] = 1e-8
    mixed[pick > 0.95] = 0.0
    w.alpha[:, 2] = mixed
    check(lib, w, plain_gate=False)


def test_gdn_bwd_rejects_a_short_workspace(lib):
    w = workloads.gdn(1, 2, 130, 16, 16, seed=3, h0=False)
    alpha, b, v, c, dout = (t.to(DEV) for t in (w.alpha, w.b, w.v, w.c, w.dout))
    _, ck = lib.gdn_fwd(alpha, b, v, c)
    need = lib.gdn_workspace_bytes(1, 2, 130, 16, 16)
    # one 16 x 16 matrix and one gate product per 32-step chunk: 2 heads x 5 chunks
    assert need == 4 * (2 * 5 * 16 * 16 + 12)
    with pytest.raises(ValueError):
        lib.gdn_bwd(alpha, b, v, c, ck, dout,
                    workspace=torch.empty(need - 16, dtype=torch.uint8, device=DEV))
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    got = lib.gdn_bwd(alpha, b, v, c, ck, dout, workspace=ws)
    ref = lib.gdn_bwd(alpha, b, v, c, ck, dout)
    torch.cuda.synchronize()
    for x, y in zip(got, ref):
        assert torch.equal(x, y)


def test_gdn_fwd_rejects_a_short_workspace(lib):
    w = workloads.gdn(1, 2, 70, 32, 16, seed=4, h0=True)
    alpha, b, v, c = (t.to(DEV) for t in (w.alpha, w.b, w.v, w.c))
    h0 = w.h0.to(DEV)
    need = lib.gdn_workspace_bytes(1, 2, 70, 32, 16)
    with pytest.raises(ValueError):
        lib.gdn_fwd(alpha, b, v, c, h0, workspace=torch.empty(need - 16, dtype=torch.uint8,
                                                             device=DEV))
    o1, k1 = lib.gdn_fwd(alpha, b, v, c, h0, workspace=torch.empty(need, dtype=torch.uint8,
                                                                   device=DEV))
    o2, k2 = lib.gdn_fwd(alpha, b, v, c, h0)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(k1, k2)


def test_gdn_on_a_side_stream(lib):
    """A caller's own stream: the same results bit for bit as on the current
    stream, with the scratch workspace the binding allocates kept alive until
    the side stream's kernels are done."""
    w = workloads.gdn(2, 4, 300, 32, 32, seed=11, h0=True)
    alpha, b, v, c, dout, h0 = (t.to(DEV) for t in (w.alpha, w.b, w.v, w.c, w.dout, w.h0))
    o_ref, ck_ref = lib.gdn_fwd(alpha, b, v, c, h0)
    g_ref = lib.gdn_bwd(alpha, b, v, c, ck_ref, dout)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    for _ in range(3):  # later calls reuse memory the allocator got back
        o, ck = lib.gdn_fwd(alpha, b, v, c, h0, stream=side)
        g = lib.gdn_bwd(alpha, b, v, c, ck, dout, stream=side)
    side.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(ck, ck_ref)
    for got, ref in zip(g, g_ref):
        assert torch.equal(got, ref)
