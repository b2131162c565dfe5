"""GPU parity of the fused RG-LRU gate preparation and scan against the fp64
oracle ("Our RG-LRU GPU audit", Strengthened fused path and Exact real chunk
algebra; the gate formulas are the method's own), through the C ABI.

Tolerance, fp32: 1e-5 of max(1, |ref|, S) per element, S the sum of the
magnitudes of the element's terms. The gates near 1 give memories of tens of
thousands of steps (a = 0.99996 at a_param = 9), and h, dx, dgate_x and dh0 are
sums over them with nonnegative weights: S is the oracle run on |x|, |dh| and
|h0| (a plain fp32 loop over such a row misses max(1, |ref|) by 2.3e-5; the
kernels, 1.8e-5). da_param sums B * T terms per channel: S from the oracle's
own dgate_a (each da_param term is dgate_a divided by log(sigmoid(a_param))
(1 - r)). dgate_a, whose terms differ in sign, keeps max(1, |ref|). With bf16
inputs (the oracle reads the same bf16 values) dx, dgate_a and dgate_x are
stored in bf16 and held to 1e-2; the fp32 outputs keep 1e-5.
"""

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from _sweep import as_f64, max_rel, sweep, worst
from associative_affine_scan_gb300 import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
TOL = 1e-5
TOLBF = 1e-2  # gradients stored in bf16 (one rounding of 2^-9)
GRADS_IN_DTYPE = ("dx", "dgate_a", "dgate_x")


def within(errs, dtype):
    """Every error within its gate: 1e-5, or 1e-2 for gradients stored in bf16."""
    return all(v <= (TOLBF if dtype == torch.bfloat16 and k in GRADS_IN_DTYPE else TOL)
               for k, v in errs.items())


def dap_scale(ga, ap, dga_ref, seg):
    """Sum over (b, t) of |the da_param terms| per channel (reset steps have
    none): |dgate_a / (log(sigmoid(a_param)) (1 - r))| sigmoid(-a_param)."""
    ga = as_f64(ga)
    ap = as_f64(ap)
    r = expit(ga)
    ls = np.log(expit(ap))[None, :, None]
    den = ls * (1.0 - r)
    # where r(1 - r) or log(sigmoid(a_param)) is 0 in fp64 the term cannot be
    # read back from dgate_a; it counts as 0 (a smaller scale: a stricter gate)
    safe = np.where(den == 0.0, 1.0, den)
    term = np.where(den == 0.0, 0.0, np.abs(np.asarray(dga_ref) / safe))
    if seg is not None:
        term = np.where((as_f64(seg) == 0)[:, None, :], 0.0, term)
    return term.sum(axis=(0, 2)) * expit(-ap)


def run(lib, w, shift=0):
    """Forward and backward on the GPU (inputs optionally shifted by `shift`
    floats off 16-byte alignment); returns host copies."""
    def dev(t):
        if t is None:
            return None
        if shift == 0:
            return t.to(DEV)
        buf = torch.empty(t.numel() + shift, dtype=t.dtype, device=DEV)
        v = buf[shift:].view(t.shape)
        v.copy_(t)
        return v
    x, ga, gx, ap, dh = (dev(t) for t in (w.x, w.gate_a, w.gate_x, w.a_param, w.dh))
    seg, h0 = dev(w.segment_pos), dev(w.h0)
    h = lib.rglru_fwd(x, ga, gx, ap, seg, h0)
    g = lib.rglru_bwd(x, ga, gx, ap, h, dh, seg, h0)
    torch.cuda.synchronize()
    return h.cpu(), [t.cpu() for t in g]


def ab(t):
    return None if t is None else t.abs()


def reference(x, ga, gx, ap, dh, seg, h0):
    """The oracle's outputs and the term scales S of h, dx, dgate_x, dh0."""
    ref_h = oracle.rglru_fwd(x, ga, gx, ap, seg, h0)
    ref_g = oracle.rglru_bwd(x, ga, gx, ap, dh, seg, h0)
    sc_h = oracle.rglru_fwd(ab(x), ga, gx, ap, seg, ab(h0))
    sc_g = oracle.rglru_bwd(ab(x), ga, gx, ap, ab(dh), seg, ab(h0))
    return ref_h, ref_g, sc_h, sc_g


def errors(h, g, ref_h, ref_g, sc_h, sc_g, dap_sc=None):
    dx, dga, dgx, dap, dh0 = g
    rdx, rdga, rdgx, rdap, rdh0 = ref_g
    errs = {"h": max_rel(h, ref_h, sc_h), "dx": max_rel(dx, rdx, sc_g[0]),
            "dgate_a": max_rel(dga, rdga), "dgate_x": max_rel(dgx, rdgx, sc_g[2]),
            "dh0": max_rel(dh0, rdh0, sc_g[4])}
    if dap_sc is not None:
        errs["da_param"] = max_rel(dap, rdap, dap_sc)
    return errs


def compare(w, h, g):
    ref_h, ref_g, sc_h, sc_g = reference(w.x, w.gate_a, w.gate_x, w.a_param, w.dh,
                                         w.segment_pos, w.h0)
    return errors(h, g, ref_h, ref_g, sc_h, sc_g,
                  dap_scale(w.gate_a, w.a_param, ref_g[1], w.segment_pos))


@pytest.mark.parametrize("T", [1, 3, 4, 5, 127, 128, 129, 257, 1000])
@pytest.mark.parametrize("B,C", [(1, 1), (3, 5), (9, 2)])
@pytest.mark.parametrize("docs", [None, (1, 60)])
def test_rglru_shapes(lib, B, C, T, docs):
    """Chunk edges (128 steps), ragged tails, one to nine rows per channel (the
    block's warps loop over more rows than they are), with and without resets
    and an initial state."""
    w = workloads.rglru(B, C, T, seed=B * 1000 + C * 10 + T, docs=docs, h0=True)
    for h0 in (w.h0, None):
        w.h0 = h0
        h, g = run(lib, w)
        errs = compare(w, h, g)
        assert within(errs, w.x.dtype), errs


@pytest.mark.parametrize("shift", [1, 2])
def test_rglru_unaligned_inputs_take_the_scalar_path(lib, shift):
    """Rows off 16-byte alignment (and T % 4 != 0) load one value at a time."""
    for T in (64, 130):
        w = workloads.rglru(2, 3, T, seed=T + shift, docs=(1, 40), h0=True)
        h, g = run(lib, w, shift=shift)
        errs = compare(w, h, g)
        assert within(errs, w.x.dtype), errs


@pytest.mark.parametrize("T", [5, 128, 129, 1000])
@pytest.mark.parametrize("docs", [None, (1, 60)])
def test_rglru_bf16_inputs(lib, T, docs):
    """x and the gate logits in bf16 (read into fp32 registers; the oracle reads
    the same bf16 values); h, da_param, dh0 in fp32, the other gradients in bf16;
    vector and one-element-off rows."""
    w = workloads.rglru(3, 5, T, seed=T + 77, docs=docs, h0=True, dtype=torch.bfloat16)
    for shift in (0, 1):
        h, g = run(lib, w, shift=shift)
        assert g[0].dtype == torch.bfloat16 and h.dtype == torch.float32
        errs = compare(w, h, g)
        assert within(errs, torch.bfloat16), errs


def test_rglru_gate_extremes(lib):
    """Frozen gates (gate_a = -30: a = 1 to fp32, multiplier near 0), open
    ones (a_param = -30: a ~ e^-100, h = sigmoid(gate_x) x), a_param = +30
    (a = 1 - O(1e-12): the clipped square root), large logits either way."""
    w = workloads.rglru(2, 4, 300, seed=7, docs=(1, 80), h0=True)
    w.gate_a[:, 0] = -30.0
    w.a_param[1] = -30.0
    w.a_param[2] = 30.0
    w.gate_x[:, 3] *= 20.0
    w.gate_a[:, 3] *= 20.0
    h, g = run(lib, w)
    errs = compare(w, h, g)
    assert all(np.isfinite(as_f64(t)).all() for t in [h] + g)
    assert all(v <= TOL for v in errs.values()), errs


@pytest.mark.parametrize("T", [256, 300, 515])
def test_rglru_resets_at_chunk_edges(lib, T):
    """Resets at the steps either side of the 128-step chunk edges, at the
    last step, and at t = 0 in one batch row (h0 erased there, dh0 = 0)."""
    w = workloads.rglru(2, 3, T, seed=T + 9, docs=None, h0=True)
    seg = torch.arange(1, T + 1, dtype=torch.int32).repeat(2, 1)
    for t in (1, 127, 128, 129, 255, 256, T - 1):
        if t < T:
            seg[0, t] = 0
    seg[1, 0] = 0
    w.segment_pos = seg
    h, g = run(lib, w)
    errs = compare(w, h, g)
    assert all(v <= TOL for v in errs.values()), errs
    assert torch.all(g[4][1] == 0.0)  # dh0 of the row that resets at t = 0


def test_rglru_full_4k_all_rows(lib):
    """Every output of the 8 x 1536 x 4096 RG-LRU workload (documents of
    512..8192 steps) against the oracle, channel batches per batch row."""
    w = workloads.rglru_4k(seed=0)
    B, C, T = w.x.shape
    h, (dx, dga, dgx, dap, dh0) = run(lib, w)
    per = 96
    nb = C // per

    def check(i0, i1):
        out = {}
        for i in range(i0, i1):
            b, c0 = divmod(i, nb)
            c0 *= per
            sl = lambda t: t[b:b + 1, c0:c0 + per]
            seg = w.segment_pos[b:b + 1]
            ap = w.a_param[c0:c0 + per]
            ref_h, rg, sc_h, sc_g = reference(sl(w.x), sl(w.gate_a), sl(w.gate_x), ap,
                                              sl(w.dh), seg, None)
            e = errors(sl(h), (sl(dx), sl(dga), sl(dgx), None, dh0[b:b + 1, c0:c0 + per]),
                       ref_h, rg, sc_h, sc_g)
            for k, v in e.items():
                out[k] = worst(out.get(k, 0.0), v)
            out[f"dap_{b}_{c0}"] = rg[3]
            out[f"dsc_{b}_{c0}"] = dap_scale(sl(w.gate_a), ap, rg[1], seg)
        return out

    # the oracle's per-batch-row da_param partials are summed over b here
    parts = {}
    errs = {}

    def wrapped(i0, i1):
        r = check(i0, i1)
        e = {k: v for k, v in r.items() if not k.startswith(("dap_", "dsc_"))}
        parts.update({k: v for k, v in r.items() if k.startswith(("dap_", "dsc_"))})
        return e

    errs = sweep(B * nb, 4, wrapped)
    ref_dap = np.zeros(C)
    scale = np.zeros(C)
    for b in range(B):
        for j in range(nb):
            ref_dap[j * per:(j + 1) * per] += parts[f"dap_{b}_{j * per}"]
            scale[j * per:(j + 1) * per] += parts[f"dsc_{b}_{j * per}"]
    errs["da_param"] = max_rel(dap, ref_dap, scale)
    print("rglru_4k all rows", errs)
    assert errs["items"] == B * nb
    assert all(errs[k] <= TOL for k in ("h", "dx", "dgate_a", "dgate_x", "dh0", "da_param")), errs
