"""Pins for the fp64 oracle, independent of the oracle's own loops.

Each test checks the oracle against something the source pages or plain
mathematics fix, so that a dropped term, a wrong sign, a wrong index or a
transposed operand in oracle.c fails at least one of them:

* exact rational brute force of the closed form
  h_t = (prod_{r<=t} a_r) h0 + sum_s (prod_{s<r<=t} a_r) x_s  (Fractions);
* the constant-gate geometric series;
* reset erasure (a_t = 0) and no leakage across packed sequences
  ("associative_scan_triton" README, how it works);
* central differences of the forward for every gradient (the loss is affine in
  each single a_t, x_t, A_t, B_t, so central differences are exact up to
  rounding) and the adjoint dot-product identity;
* log space against the linear scan and against torch.logcumsumexp;
* the block form against k = 1, diagonal A, A = I (numpy cumsum) and explicit
  numpy matrix products;
* the chunk algebra of "Our RG-LRU GPU audit" (Exact real chunk algebra)
  composed in random bracketings;
* the RG-LRU gate preparation (the same page, Strengthened fused path):
  the transition against sigmoid(a_param)^(8 r) from a library sigmoid, the
  multiplier against a^2 + mult^2 = 1, frozen and open gates, the whole
  sequence against the pinned scalar scan of its one-step maps, reset
  erasure, and central differences for every gradient.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# exact closed forms
# ---------------------------------------------------------------------------

def closed_form_fwd(a, x, h0):
    """Exact h_t from the sum-of-products closed form (no recurrence)."""
    a = [Fraction(float(v)) for v in a]
    x = [Fraction(float(v)) for v in x]
    h0 = Fraction(float(h0))
    T = len(a)
    out = []
    for t in range(T):
        prod_all = Fraction(1)
        for r in range(t + 1):
            prod_all *= a[r]
        acc = prod_all * h0
        for s in range(t + 1):
            p = Fraction(1)
            for r in range(s + 1, t + 1):
                p *= a[r]
            acc += p * x[s]
        out.append(acc)
    return out


def closed_form_dx(a, dh):
    """Exact dL/dx_t = sum_{s>=t} (prod_{t<r<=s} a_r) dh_s (no recurrence)."""
    a = [Fraction(float(v)) for v in a]
    dh = [Fraction(float(v)) for v in dh]
    T = len(a)
    out = []
    for t in range(T):
        acc = Fraction(0)
        for s in range(t, T):
            p = Fraction(1)
            for r in range(t + 1, s + 1):
                p *= a[r]
            acc += p * dh[s]
        out.append(acc)
    return out


@pytest.mark.parametrize("seed", range(4))
def test_fwd_matches_exact_closed_form(seed):
    g = rng(seed)
    T = 11
    a = g.uniform(-1.2, 1.2, size=(1, 1, T))
    x = g.normal(size=(1, 1, T))
    h0 = g.normal(size=(1, 1))
    h = oracle.scan_fwd(a, x, h0)
    exact = closed_form_fwd(a[0, 0], x[0, 0], h0[0, 0])
    for t in range(T):
        assert abs(h[0, 0, t] - float(exact[t])) <= 1e-13 * max(1.0, abs(float(exact[t])))


def test_fwd_reverse_matches_closed_form_on_flipped_input():
    g = rng(7)
    T = 9
    a = g.uniform(0, 1, size=(1, 1, T))
    x = g.normal(size=(1, 1, T))
    h0 = g.normal(size=(1, 1))
    h = oracle.scan_fwd(a, x, h0, reverse=True)
    exact = closed_form_fwd(a[0, 0, ::-1], x[0, 0, ::-1], h0[0, 0])[::-1]
    for t in range(T):
        assert abs(h[0, 0, t] - float(exact[t])) <= 1e-13 * max(1.0, abs(float(exact[t])))


@pytest.mark.parametrize("c", [0.5, 0.9, -0.75, 1.0])
def test_constant_gate_geometric_series(c):
    T = 40
    xv, h0v = 0.3, -1.7
    a = np.full((1, 1, T), c)
    x = np.full((1, 1, T), xv)
    h = oracle.scan_fwd(a, x, np.array([[h0v]]))[0, 0]
    t = np.arange(T) + 1
    if c == 1.0:
        ref = h0v + t * xv
    else:
        ref = c ** t * h0v + xv * (1 - c ** t) / (1 - c)
    np.testing.assert_allclose(h, ref, rtol=1e-13, atol=1e-13)


def test_reset_erases_prefix_exactly():
    g = rng(3)
    T = 50
    a = g.uniform(0, 1, size=(2, 3, T))
    x = g.normal(size=(2, 3, T))
    a[..., 20] = 0.0
    h = oracle.scan_fwd(a, x, g.normal(size=(2, 3)))
    assert np.array_equal(h[..., 20], x[..., 20])
    # perturbing anything before the reset leaves the outputs from it on unchanged
    a2, x2 = a.copy(), x.copy()
    a2[..., :20] = g.uniform(0, 1, size=(2, 3, 20))
    x2[..., :20] = g.normal(size=(2, 3, 20))
    h2 = oracle.scan_fwd(a2, x2, g.normal(size=(2, 3)))
    assert np.array_equal(h[..., 20:], h2[..., 20:])
    assert not np.array_equal(h[..., :20], h2[..., :20])


def segments_as_dense(a, x, h0, cu, reverse):
    out = np.zeros_like(a)
    for s in range(len(cu) - 1):
        b, e = cu[s], cu[s + 1]
        if e == b:
            continue
        seg = oracle.scan_fwd(a[None, :, b:e], x[None, :, b:e],
                              None if h0 is None else h0[s][None, :], reverse=reverse)
        out[:, b:e] = seg[0]
    return out


@pytest.mark.parametrize("reverse", [False, True])
def test_packed_sequences_do_not_leak(reverse):
    g = rng(11)
    cu = np.array([0, 5, 5, 17, 18, 30], dtype=np.int32)  # includes an empty segment
    C, T = 3, int(cu[-1])
    a = g.uniform(0, 1, size=(C, T))
    x = g.normal(size=(C, T))
    h0 = g.normal(size=(len(cu) - 1, C))
    h = oracle.scan_fwd(a, x, h0, cu_seqlens=cu, reverse=reverse)
    ref = segments_as_dense(a, x, h0, cu, reverse)
    assert np.array_equal(h, ref)
    # perturbing segment 2 leaves the others bit-identical
    a2 = a.copy()
    a2[:, 5:17] = g.uniform(0, 1, size=(C, 12))
    h2 = oracle.scan_fwd(a2, x, h0, cu_seqlens=cu, reverse=reverse)
    keep = np.r_[0:5, 17:30]
    assert np.array_equal(h[:, keep], h2[:, keep])


def test_stream_continuation():
    g = rng(5)
    T = 64
    a = g.uniform(0, 1.1, size=(2, 2, T))
    x = g.normal(size=(2, 2, T))
    h0 = g.normal(size=(2, 2))
    whole = oracle.scan_fwd(a, x, h0)
    split = 23
    first = oracle.scan_fwd(a[..., :split], x[..., :split], h0)
    second = oracle.scan_fwd(a[..., split:], x[..., split:], first[..., -1])
    np.testing.assert_allclose(np.concatenate([first, second], -1), whole, rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------------------
# scalar backward
# ---------------------------------------------------------------------------

def loss_scalar(a, x, h0, dh, cu=None, reverse=False):
    return float(np.sum(oracle.scan_fwd(a, x, h0, cu_seqlens=cu, reverse=reverse) * dh))


@pytest.mark.parametrize("reverse", [False, True])
def test_bwd_central_differences(reverse):
    g = rng(21 + reverse)
    B, C, T = 1, 2, 13
    a = g.uniform(-1, 1, size=(B, C, T))
    x = g.normal(size=(B, C, T))
    h0 = g.normal(size=(B, C))
    dh = g.normal(size=(B, C, T))
    da, dx, dh0 = oracle.scan_bwd(a, x, dh, h0, reverse=reverse)
    eps = 1e-5
    for arr, grad in ((a, da), (x, dx), (h0, dh0)):
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss_scalar(a, x, h0, dh, reverse=reverse)
            arr[idx] = old - eps
            lm = loss_scalar(a, x, h0, dh, reverse=reverse)
            arr[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-8 * max(1.0, abs(fd)), (idx, fd, grad[idx])


def test_bwd_dx_matches_exact_closed_form():
    g = rng(31)
    T = 10
    a = g.uniform(-1, 1, size=(1, 1, T))
    x = g.normal(size=(1, 1, T))
    dh = g.normal(size=(1, 1, T))
    _, dx, _ = oracle.scan_bwd(a, x, dh)
    exact = closed_form_dx(a[0, 0], dh[0, 0])
    for t in range(T):
        assert abs(dx[0, 0, t] - float(exact[t])) <= 1e-13 * max(1.0, abs(float(exact[t])))


def test_bwd_adjoint_identity():
    # h is linear in (x, h0) for fixed a: <dh, J dx_dir> = <dx, dx_dir> + <dh0, dh0_dir>
    g = rng(41)
    B, C, T = 2, 3, 37
    a = g.uniform(0, 1, size=(B, C, T))
    x = g.normal(size=(B, C, T))
    h0 = g.normal(size=(B, C))
    dh = g.normal(size=(B, C, T))
    _, dx, dh0 = oracle.scan_bwd(a, x, dh, h0)
    vx = g.normal(size=(B, C, T))
    v0 = g.normal(size=(B, C))
    jv = oracle.scan_fwd(a, vx, v0)  # J applied to the direction (x, h0 enter linearly)
    lhs = float(np.sum(dh * jv))
    rhs = float(np.sum(dx * vx) + np.sum(dh0 * v0))
    assert abs(lhs - rhs) <= 1e-11 * max(1.0, abs(lhs))


@pytest.mark.parametrize("reverse", [False, True])
def test_bwd_packed_central_differences_and_boundaries(reverse):
    g = rng(51 + reverse)
    cu = np.array([0, 4, 4, 9, 10, 15], dtype=np.int32)
    C, T = 2, int(cu[-1])
    a = g.uniform(-1, 1, size=(C, T))
    x = g.normal(size=(C, T))
    h0 = g.normal(size=(len(cu) - 1, C))
    dh = g.normal(size=(C, T))
    da, dx, dh0 = oracle.scan_bwd(a, x, dh, h0, cu_seqlens=cu, reverse=reverse)
    eps = 1e-5
    for arr, grad in ((a, da), (x, dx), (h0, dh0)):
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss_scalar(a, x, h0, dh, cu, reverse)
            arr[idx] = old - eps
            lm = loss_scalar(a, x, h0, dh, cu, reverse)
            arr[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-8 * max(1.0, abs(fd)), (idx, fd, grad[idx])
    # the last step of every segment (in scan direction) has d_tokens == dh exactly
    for s in range(len(cu) - 1):
        b, e = cu[s], cu[s + 1]
        if e > b:
            last = b if reverse else e - 1
            assert np.array_equal(dx[:, last], dh[:, last])
    assert np.all(dh0[1] == 0.0)  # the empty segment


# ---------------------------------------------------------------------------
# log space
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("reverse", [False, True])
def test_log_matches_linear_scan(reverse):
    g = rng(61)
    B, C, T = 2, 3, 200
    la = np.log(torch.sigmoid(torch.from_numpy(g.normal(size=(B, C, T)))).numpy())
    lx = g.normal(size=(B, C, T))
    lh0 = g.normal(size=(B, C))
    h = oracle.scan_log_fwd(la, lx, lh0, reverse=reverse)
    ref = oracle.scan_fwd(np.exp(la), np.exp(lx), np.exp(lh0), reverse=reverse)
    np.testing.assert_allclose(h, ref, rtol=1e-12, atol=0)


def test_log_matches_logcumsumexp_closed_form():
    # l_t = S_t + logcumsumexp(lx - S)_t, S = cumsum(la), no initial state
    g = rng(62)
    T = 64
    la = -g.uniform(0.0, 0.5, size=(1, 2, T))
    lx = g.normal(size=(1, 2, T))
    h = oracle.scan_log_fwd(la, lx)
    S = torch.from_numpy(la).cumsum(-1)
    ell = S + torch.logcumsumexp(torch.from_numpy(lx) - S, dim=-1)
    np.testing.assert_allclose(h, torch.exp(ell).numpy(), rtol=1e-12, atol=0)


def test_log_reset_and_packed():
    g = rng(63)
    cu = np.array([0, 7, 20], dtype=np.int32)
    la = -g.uniform(0, 1, size=(2, 20))
    lx = g.normal(size=(2, 20))
    la[:, 12] = -np.inf  # a_t = 0
    lh0 = g.normal(size=(2, 2))
    h = oracle.scan_log_fwd(la, lx, lh0, cu_seqlens=cu)
    ref = oracle.scan_fwd(np.exp(la), np.exp(lx), np.exp(lh0), cu_seqlens=cu)
    np.testing.assert_allclose(h, ref, rtol=1e-12, atol=0)
    np.testing.assert_allclose(h[:, 12], np.exp(lx[:, 12]), rtol=1e-15)


def test_log_bwd_central_differences():
    g = rng(64)
    B, C, T = 1, 2, 9
    la = -g.uniform(0.1, 1, size=(B, C, T))
    lx = g.normal(size=(B, C, T))
    lh0 = g.normal(size=(B, C))
    dh = g.normal(size=(B, C, T))
    dla, dlx, dlh0 = oracle.scan_log_bwd(la, lx, dh, lh0)

    def loss():
        return float(np.sum(oracle.scan_log_fwd(la, lx, lh0) * dh))

    eps = 1e-6
    for arr, grad in ((la, dla), (lx, dlx), (lh0, dlh0)):
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss()
            arr[idx] = old - eps
            lm = loss()
            arr[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, grad[idx])


# ---------------------------------------------------------------------------
# block-matrix affine form
# ---------------------------------------------------------------------------

def test_affine_k1_is_scalar_scan():
    g = rng(71)
    B, T, N = 2, 30, 3
    A = g.uniform(-1, 1, size=(B, T, N, 1, 1))
    Bm = g.normal(size=(B, T, N, 1, 1))
    h0 = g.normal(size=(B, N, 1, 1))
    H = oracle.affine_fwd(A, Bm, h0)
    # scalar layout [B, C=N, T]
    a = A[..., 0, 0].transpose(0, 2, 1)
    x = Bm[..., 0, 0].transpose(0, 2, 1)
    h = oracle.scan_fwd(a, x, h0[..., 0, 0])
    np.testing.assert_allclose(H[..., 0, 0].transpose(0, 2, 1), h, rtol=1e-14, atol=1e-14)


def test_affine_diagonal_is_independent_scalar_scans():
    g = rng(72)
    B, T, N, k, v = 1, 25, 2, 3, 2
    d = g.uniform(-1, 1, size=(B, T, N, k))
    A = np.zeros((B, T, N, k, k))
    for i in range(k):
        A[..., i, i] = d[..., i]
    Bm = g.normal(size=(B, T, N, k, v))
    h0 = g.normal(size=(B, N, k, v))
    H = oracle.affine_fwd(A, Bm, h0)
    for i in range(k):
        for j in range(v):
            h = oracle.scan_fwd(d[..., i].transpose(0, 2, 1), Bm[..., i, j].transpose(0, 2, 1),
                                h0[..., i, j])
            np.testing.assert_allclose(H[..., i, j].transpose(0, 2, 1), h, rtol=1e-14, atol=1e-14)


def test_affine_identity_is_cumsum():
    g = rng(73)
    B, T, N, k, v = 2, 17, 2, 4, 3
    A = np.broadcast_to(np.eye(k), (B, T, N, k, k)).copy()
    Bm = g.normal(size=(B, T, N, k, v))
    H = oracle.affine_fwd(A, Bm)
    np.testing.assert_allclose(H, np.cumsum(Bm, axis=1), rtol=1e-13, atol=1e-13)


def test_affine_explicit_products_and_order():
    g = rng(74)
    B, T, N, k, v = 1, 6, 1, 3, 2
    A = g.normal(size=(B, T, N, k, k))
    Bm = g.normal(size=(B, T, N, k, v))
    h0 = g.normal(size=(B, N, k, v))
    H = oracle.affine_fwd(A, Bm, h0)
    for t in range(T):
        acc = np.eye(k)
        for r in range(t + 1):
            acc = A[0, r, 0] @ acc  # A_t ... A_0
        ref = acc @ h0[0, 0]
        for s in range(t + 1):
            p = np.eye(k)
            for r in range(s + 1, t + 1):
                p = A[0, r, 0] @ p
            ref = ref + p @ Bm[0, s, 0]
        np.testing.assert_allclose(H[0, t, 0], ref, rtol=1e-12, atol=1e-12)
    # the product order matters: the reversed product A_0 ... A_t differs
    wrong = np.eye(k)
    for r in range(T):
        wrong = wrong @ A[0, r, 0]
    right = np.eye(k)
    for r in range(T):
        right = A[0, r, 0] @ right
    assert not np.allclose(wrong @ h0[0, 0], right @ h0[0, 0])


def test_affine_bwd_central_differences():
    g = rng(75)
    B, T, N, k, v = 1, 5, 2, 3, 2
    A = g.normal(size=(B, T, N, k, k)) * 0.7
    Bm = g.normal(size=(B, T, N, k, v))
    h0 = g.normal(size=(B, N, k, v))
    dH = g.normal(size=(B, T, N, k, v))
    dA, dB, dh0 = oracle.affine_bwd(A, Bm, dH, h0)

    def loss():
        return float(np.sum(oracle.affine_fwd(A, Bm, h0) * dH))

    eps = 1e-5
    for arr, grad in ((A, dA), (Bm, dB), (h0, dh0)):
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss()
            arr[idx] = old - eps
            lm = loss()
            arr[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-8 * max(1.0, abs(fd)), (idx, fd, grad[idx])


# ---------------------------------------------------------------------------
# chunk algebra
# ---------------------------------------------------------------------------

def test_chunk_summaries_compose_in_any_bracketing():
    g = rng(81)
    T = 97
    a = g.uniform(-1, 1, size=T)
    x = g.normal(size=T)
    h0 = 0.37
    whole = oracle.scan_fwd(a[None, None], x[None, None], np.array([[h0]]))[0, 0, -1]
    for trial in range(10):
        cuts = np.sort(g.choice(np.arange(1, T), size=6, replace=False))
        bounds = np.r_[0, cuts, T]
        sums = [oracle.chunk_summary(a[b:e], x[b:e]) for b, e in zip(bounds[:-1], bounds[1:])]
        # random bracketing: repeatedly compose a random adjacent pair
        while len(sums) > 1:
            i = int(g.integers(0, len(sums) - 1))
            sums[i:i + 2] = [oracle.compose(sums[i], sums[i + 1])]
        P, Q = sums[0]
        assert abs(P * h0 + Q - whole) <= 1e-12 * max(1.0, abs(whole))


def test_compose_identity_and_order():
    s = (0.5, 2.0)
    assert oracle.compose((1.0, 0.0), s) == s
    assert oracle.compose(s, (1.0, 0.0)) == s
    # "apply (0.5, 2) then (3, 1)": h -> 3 (0.5 h + 2) + 1 = 1.5 h + 7
    assert oracle.compose((0.5, 2.0), (3.0, 1.0)) == (1.5, 7.0)
    assert oracle.compose((3.0, 1.0), (0.5, 2.0)) == (1.5, 2.5)
    # a reset (P = 0) erases the earlier summary
    assert oracle.compose((0.7, -4.0), (0.0, 3.0)) == (0.0, 3.0)


def test_affine_coefficient_prefix_is_the_product_of_gates():
    """Abar_t = A_t ... A_0 ("Triton scan kernels", One associative-scan family:
    the composed coefficient) equals the block scan with B = 0 and h0 = I;
    checked against explicit numpy products, later factors on the left."""
    g = np.random.default_rng(4)
    B, T, N, k = 1, 6, 2, 3
    A = g.standard_normal((B, T, N, k, k)) * 0.7
    eye = np.broadcast_to(np.eye(k), (B, N, k, k)).copy()
    got = oracle.affine_fwd(A, np.zeros_like(A), eye)
    for n in range(N):
        P = np.eye(k)
        for t in range(T):
            P = A[0, t, n] @ P
            assert np.allclose(got[0, t, n], P, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------
# scalar-gated outer-product state ("Operations & Triton Kernels" (HyMo))
# ---------------------------------------------------------------------------

def _gdn_inputs(g, B, H, T, S, D, dyadic=False):
    if dyadic:
        al = g.choice([0.0, 0.5, 1.0, 0.25], size=(B, H, T))
        b = g.integers(-3, 4, size=(B, H, T, S)).astype(np.float64)
        v = g.integers(-3, 4, size=(B, H, T, D)).astype(np.float64)
        c = g.integers(-3, 4, size=(B, H, T, S)).astype(np.float64)
        h0 = g.integers(-3, 4, size=(B, H, S, D)).astype(np.float64)
    else:
        al = g.random((B, H, T))
        b, c = g.standard_normal((B, H, T, S)), g.standard_normal((B, H, T, S))
        v, h0 = g.standard_normal((B, H, T, D)), g.standard_normal((B, H, S, D))
    return al, b, v, c, h0


def test_gdn_forward_exact_closed_form():
    """h_t = (prod_{r<=t} alpha_r) h0 + sum_{u<=t} (prod_{u<r<=t} alpha_r) b_u v_u^T and
    o_t = h_t^T c_t, in exact rational arithmetic (dyadic inputs: every fp64
    partial result is exact, so the oracle must match bit for bit)."""
    g = np.random.default_rng(11)
    B, H, T, S, D = 1, 2, 5, 3, 2
    al, b, v, c, h0 = _gdn_inputs(g, B, H, T, S, D, dyadic=True)
    got = oracle.gdn_fwd(al, b, v, c, h0)
    F = Fraction
    for hh in range(H):
        for t in range(T):
            for d in range(D):
                o = F(0)
                for s_ in range(S):
                    prod = F(1)
                    for r in range(t + 1):
                        prod *= F(al[0, hh, r])
                    h = prod * F(h0[0, hh, s_, d])
                    for u in range(t + 1):
                        w = F(1)
                        for r in range(u + 1, t + 1):
                            w *= F(al[0, hh, r])
                        h += w * F(b[0, hh, u, s_]) * F(v[0, hh, u, d])
                    o += F(c[0, hh, t, s_]) * h
                assert got[0, hh, t, d] == float(o)


def test_gdn_with_one_by_one_state_is_the_scalar_scan():
    """S = D = 1: h_t = alpha_t h_{t-1} + b_t v_t, o_t = c_t h_t."""
    g = np.random.default_rng(12)
    al, b, v, c, h0 = _gdn_inputs(g, 2, 3, 40, 1, 1)
    got = oracle.gdn_fwd(al, b, v, c, h0)
    h = oracle.scan_fwd(torch.tensor(al), torch.tensor(b[..., 0] * v[..., 0]),
                        torch.tensor(h0[..., 0, 0]))
    assert np.allclose(got[..., 0], c[..., 0] * np.asarray(h), rtol=1e-14, atol=1e-14)


def test_gdn_backward_central_differences():
    """L = sum <do, o> is linear in b, v, c and h0 separately (central differences
    are exact up to rounding) and polynomial in alpha (O(eps^2))."""
    g = np.random.default_rng(13)
    B, H, T, S, D = 1, 2, 6, 3, 2
    al, b, v, c, h0 = _gdn_inputs(g, B, H, T, S, D)
    do = g.standard_normal((B, H, T, D))
    dal, db, dv, dc, dh0 = oracle.gdn_bwd(al, b, v, c, do, h0)

    def loss(al_, b_, v_, c_, h0_):
        return float((oracle.gdn_fwd(al_, b_, v_, c_, h0_) * do).sum())

    args = [al, b, v, c, h0]
    for which, grad, eps, tol in ((0, dal, 1e-5, 1e-8), (1, db, 1e-3, 1e-9), (2, dv, 1e-3, 1e-9),
                                  (3, dc, 1e-3, 1e-9), (4, dh0, 1e-3, 1e-9)):
        x = args[which]
        for idx in np.ndindex(x.shape):
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            fd = (loss(*plus) - loss(*minus)) / (2 * eps)
            assert abs(fd - grad[idx]) <= tol * max(1.0, abs(fd)), (which, idx, fd, grad[idx])


# ---------------------------------------------------------------------------
# RG-LRU gate preparation ("Our RG-LRU GPU audit", Strengthened fused path and
# Exact real chunk algebra; the gate formulas are the method's own)
# ---------------------------------------------------------------------------

def _expit(z):
    from scipy.special import expit
    return expit(z)


def _rglru_inputs(g, B, C, T, resets=True):
    x = g.standard_normal((B, C, T))
    ga = g.standard_normal((B, C, T))
    gx = g.standard_normal((B, C, T))
    ap = 2.0 + g.standard_normal(C)
    h0 = g.standard_normal((B, C))
    seg = None
    if resets:
        seg = np.tile(np.arange(T, dtype=np.int32), (B, 1)) + 1
        for b in range(B):
            for t in g.choice(T, size=max(1, T // 8), replace=False):
                seg[b, t:] = np.arange(T - t, dtype=np.int32)  # a new segment starts at t
    return x, ga, gx, ap, seg, h0


def _step_maps(x, ga, gx, ap, seg):
    """a_t and write_t of every step, each read off a one-step call of the
    oracle: from h0 = 1 with x = 0 (h = a) and from h0 = 0 (h = write)."""
    B, C, T = x.shape
    a = np.empty_like(x)
    w = np.empty_like(x)
    for b in range(B):
        for t in range(T):
            reset = seg is not None and seg[b, t] == 0
            sp = np.zeros((1, 1), dtype=np.int32) if reset else None
            col = lambda arr: arr[b, :, t].reshape(1, C, 1)
            a[b, :, t] = oracle.rglru_fwd(np.zeros((1, C, 1)), col(ga), col(gx), ap, sp,
                                          np.ones((1, C)))[0, :, 0]
            w[b, :, t] = oracle.rglru_fwd(col(x), col(ga), col(gx), ap, sp,
                                          np.zeros((1, C)))[0, :, 0]
    return a, w


def test_rglru_transition_and_multiplier():
    """a = sigmoid(a_param)^(8 sigmoid(gate_a)) (the same number as
    exp(-8 softplus(-a_param) r), computed another way), and the multiplier
    closes a^2 + mult^2 = 1."""
    g = np.random.default_rng(40)
    C = 64
    ga, gx = g.standard_normal((1, C, 1)) * 3, g.standard_normal((1, C, 1)) * 3
    ap = g.standard_normal(C) * 4
    a = oracle.rglru_fwd(np.zeros((1, C, 1)), ga, gx, ap, None, np.ones((1, C)))[0, :, 0]
    want = _expit(ap) ** (8.0 * _expit(ga[0, :, 0]))
    assert np.allclose(a, want, rtol=1e-12, atol=0)
    w = oracle.rglru_fwd(np.ones((1, C, 1)), ga, gx, ap, None, np.zeros((1, C)))[0, :, 0]
    mult = w / _expit(gx[0, :, 0])
    assert (mult >= 0).all()
    assert np.allclose(a * a + mult * mult, 1.0, rtol=0, atol=1e-12)


def test_rglru_frozen_and_open_gates():
    """r -> 0 (gate_a = -80): a = 1 and the multiplier vanishes, the state
    is carried unchanged. a_param -> -inf (-80): a ~ e^-170, the multiplier is
    1 and h_t = sigmoid(gate_x_t) x_t."""
    g = np.random.default_rng(41)
    B, C, T = 2, 3, 50
    x, ga, gx, ap, _, h0 = _rglru_inputs(g, B, C, T, resets=False)
    h = oracle.rglru_fwd(x, np.full_like(ga, -80.0), gx, ap, None, h0)
    assert np.allclose(h, h0[:, :, None], rtol=1e-12, atol=1e-12)
    gb = np.clip(ga, -1.0, 1.0)
    h = oracle.rglru_fwd(x, gb, gx, np.full(C, -80.0), None, h0)
    assert np.allclose(h, _expit(gx) * x, rtol=1e-13, atol=1e-15)


def test_rglru_is_the_scan_of_its_step_maps():
    """The whole sequence equals the scalar scan (pinned above) of the step
    maps (a_t, write_t) that one-step calls give, resets included: the gates
    are read per (b, c, t), a_param per channel, segment_pos per (b, t)."""
    g = np.random.default_rng(42)
    x, ga, gx, ap, seg, h0 = _rglru_inputs(g, 2, 3, 37)
    a, w = _step_maps(x, ga, gx, ap, seg)
    got = oracle.rglru_fwd(x, ga, gx, ap, seg, h0)
    want = np.asarray(oracle.scan_fwd(torch.tensor(a), torch.tensor(w), torch.tensor(h0)))
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_rglru_reset_erases_the_prefix():
    """Where segment_pos == 0: h_t = sigmoid(gate_x_t) x_t exactly, whatever
    came before; inputs before the reset change nothing from it on."""
    g = np.random.default_rng(43)
    x, ga, gx, ap, seg, h0 = _rglru_inputs(g, 2, 3, 40)
    seg[:, 17] = 0
    h = oracle.rglru_fwd(x, ga, gx, ap, seg, h0)
    for b in range(2):
        for t in range(40):
            if seg[b, t] == 0:
                assert np.array_equal(h[b, :, t], _expit(gx[b, :, t]) * x[b, :, t])
    x2, ga2, h02 = x.copy(), ga.copy(), h0 * 3.0
    x2[:, :, :17] += 1.0
    ga2[:, :, :17] -= 2.0
    h2 = oracle.rglru_fwd(x2, ga2, gx, ap, seg, h02)
    assert np.array_equal(h2[:, :, 17:], h[:, :, 17:])


def test_rglru_backward_central_differences():
    """Every gradient of L = sum dh * h against central differences of the
    forward (smooth in each input; inputs away from the square root's clip)."""
    g = np.random.default_rng(44)
    B, C, T = 2, 2, 9
    x, ga, gx, ap, seg, h0 = _rglru_inputs(g, B, C, T, resets=False)
    seg = np.tile(np.arange(T, dtype=np.int32), (B, 1)) + 1
    seg[0, 4:] = np.arange(T - 4)  # a reset inside row 0 of each channel
    dh = g.standard_normal((B, C, T))
    dx, dga, dgx, dap, dh0 = oracle.rglru_bwd(x, ga, gx, ap, dh, seg, h0)

    def loss(*args):
        return float((oracle.rglru_fwd(args[0], args[1], args[2], args[3], seg, args[4]) * dh).sum())

    args = [x, ga, gx, ap, h0]
    for which, grad in ((0, dx), (1, dga), (2, dgx), (3, dap), (4, dh0)):
        arr = args[which]
        for idx in np.ndindex(arr.shape):
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += 1e-6
            minus[which][idx] -= 1e-6
            fd = (loss(*plus) - loss(*minus)) / 2e-6
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (which, idx, fd, grad[idx])
    # a reset's gate has no effect: its gradient is 0, and dh0 of row 0 sees
    # the steps before the reset only
    assert np.all(dga[0, :, 4] == 0.0)
