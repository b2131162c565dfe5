"""The stored dyadic worked examples under tests/golden/ against exact arithmetic.

The expected values were written by tests/golden/write_golden.py from the
oracle; here they are checked against exact rational closed forms computed
independently of the oracle (sums of products, no recurrence), and against the
oracle itself so that a later change to it cannot drift silently.
"""

import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def fr(v):
    return Fraction(float(v))


def segment_closed_form(a, x, h0, dh):
    """Exact (h, da, dx, dh0) of one causal segment from sums of products."""
    a = [fr(v) for v in a]
    x = [fr(v) for v in x]
    dh = [fr(v) for v in dh]
    h0 = fr(h0)
    T = len(a)

    def prod(lo, hi):  # prod_{lo <= r <= hi} a_r
        p = Fraction(1)
        for r in range(lo, hi + 1):
            p *= a[r]
        return p

    h = [prod(0, t) * h0 + sum(prod(s + 1, t) * x[s] for s in range(t + 1)) for t in range(T)]
    dx = [sum(prod(t + 1, s) * dh[s] for s in range(t, T)) for t in range(T)]
    da = [dx[t] * (h[t - 1] if t > 0 else h0) for t in range(T)]
    dh0 = a[0] * dx[0] if T else Fraction(0)
    return h, da, dx, dh0


def check_row(res, key, row_slice, a, x, h0, dh, reverse):
    if reverse:
        a, x, dh = a[::-1], x[::-1], dh[::-1]
    h, da, dx, dh0 = segment_closed_form(a, x, h0, dh)
    if reverse:
        h, da, dx = h[::-1], da[::-1], dx[::-1]
    for name, exact in (("h", h), ("da", da), ("dx", dx)):
        got = res[name]
        for t, e in zip(row_slice, exact):
            assert Fraction(got(t)) == e, (key, name, t)
    return dh0


@pytest.mark.parametrize("direction", ["causal", "reverse"])
def test_scalar_dense_golden_is_exact(direction):
    g = load("scalar_dense_dyadic.json")
    rev = direction == "reverse"
    res = g[direction]
    for c in range(2):
        view = {k: (lambda t, k=k, c=c: res[k][0][c][t]) for k in ("h", "da", "dx")}
        dh0 = check_row(view, direction, range(12), g["a"][0][c], g["x"][0][c], g["h0"][0][c],
                        g["dh"][0][c], rev)
        assert Fraction(res["dh0"][0][c]) == dh0


@pytest.mark.parametrize("direction", ["causal", "reverse"])
def test_scalar_packed_golden_is_exact(direction):
    g = load("scalar_packed_dyadic.json")
    rev = direction == "reverse"
    res = g[direction]
    cu = g["cu_seqlens"]
    for c in range(2):
        for s in range(len(cu) - 1):
            b, e = cu[s], cu[s + 1]
            view = {k: (lambda t, k=k, c=c: res[k][c][t]) for k in ("h", "da", "dx")}
            dh0 = check_row(view, direction, range(b, e), g["a"][c][b:e], g["x"][c][b:e],
                            g["h0"][s][c], g["dh"][c][b:e], rev)
            assert Fraction(res["dh0"][s][c]) == (dh0 if e > b else 0)


def test_affine_golden_is_exact():
    g = load("affine_2x2_dyadic.json")
    A = np.array(g["A"])
    Bm = np.array(g["Bm"])
    h0 = np.array(g["h0"])
    dH = np.array(g["dH"])
    B, T, N, k, v = Bm.shape[0], Bm.shape[1], Bm.shape[2], A.shape[3], Bm.shape[4]

    def mat(m):
        return [[fr(e) for e in row] for row in m]

    def mul(X, Y):
        return [[sum(X[i][l] * Y[l][j] for l in range(len(Y))) for j in range(len(Y[0]))]
                for i in range(len(X))]

    def add(X, Y):
        return [[X[i][j] + Y[i][j] for j in range(len(X[0]))] for i in range(len(X))]

    def tr(X):
        return [list(r) for r in zip(*X)]

    for b in range(B):
        for n in range(N):
            As = [mat(A[b, t, n]) for t in range(T)]
            Bs = [mat(Bm[b, t, n]) for t in range(T)]
            H0 = mat(h0[b, n])
            Hs = []
            for t in range(T):  # closed form: A_t..A_0 h0 + sum_s A_t..A_{s+1} B_s
                P = [[Fraction(int(i == j)) for j in range(k)] for i in range(k)]
                for r in range(t + 1):
                    P = mul(As[r], P)
                acc = mul(P, H0)
                for s in range(t + 1):
                    Ps = [[Fraction(int(i == j)) for j in range(k)] for i in range(k)]
                    for r in range(s + 1, t + 1):
                        Ps = mul(As[r], Ps)
                    acc = add(acc, mul(Ps, Bs[s]))
                Hs.append(acc)
                assert [[Fraction(e) for e in row] for row in g["H"][b][t][n]] == acc
            # adjoint: G_t = sum_{s>=t} (A_s..A_{t+1})^T dH_s
            for t in range(T):
                G = [[Fraction(0)] * v for _ in range(k)]
                for s in range(t, T):
                    Ps = [[Fraction(int(i == j)) for j in range(k)] for i in range(k)]
                    for r in range(t + 1, s + 1):
                        Ps = mul(As[r], Ps)
                    G = add(G, mul(tr(Ps), mat(dH[b, s, n])))
                assert [[Fraction(e) for e in row] for row in g["dB"][b][t][n]] == G
                prev = Hs[t - 1] if t > 0 else H0
                assert [[Fraction(e) for e in row] for row in g["dA"][b][t][n]] == mul(G, tr(prev))
                if t == 0:
                    assert [[Fraction(e) for e in row] for row in g["dh0"][b][n]] == \
                        mul(tr(As[0]), G)


def test_oracle_reproduces_golden():
    g = load("scalar_packed_dyadic.json")
    for key, rev in (("causal", False), ("reverse", True)):
        h = oracle.scan_fwd(np.array(g["a"]), np.array(g["x"]), np.array(g["h0"]),
                            cu_seqlens=np.array(g["cu_seqlens"]), reverse=rev)
        assert np.array_equal(h, np.array(g[key]["h"]))
    g = load("affine_2x2_dyadic.json")
    H = oracle.affine_fwd(np.array(g["A"]), np.array(g["Bm"]), np.array(g["h0"]))
    assert np.array_equal(H, np.array(g["H"]))
