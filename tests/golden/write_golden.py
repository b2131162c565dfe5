"""Write the small dyadic worked examples under tests/golden/.

Every stored expected value is computed here by the fp64 oracle (and nothing
else). The inputs are dyadic with short runs, so every partial result of the
recurrence is exactly representable in fp32 as well: any evaluation order gives
the same bits. test_golden.py checks the stored values against exact rational
arithmetic, and the GPU tests require bit-exact agreement.

Sources of the recurrences (page titles and sections):
* scalar: "associative_scan_triton" README, quick start (h[t] = g[t] * h[t-1]
  + x[t], cu_seqlens packing, scan_bidirectional_branched) and how it works
  (backward: reverse scan on shifted gates, d_gates = shifted_states * d_tokens);
* block: "Triton scan kernels", One associative-scan family (h_t = A_t h_{t-1}
  + B_t) and Autograd integration and the reversed-scan backward.

Run: python tests/golden/write_golden.py
"""

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def dump(name, payload):
    with open(os.path.join(HERE, name), "w") as f:
        json.dump(payload, f, indent=1)
        f.write("\n")


def scalar_dense():
    a = [[[0.5, 1.0, -1.0, 0.5, 0.0, 1.0, 0.5, 0.5, -1.0, 1.0, 0.0, 0.5],
          [1.0, 0.5, 0.5, 0.0, -1.0, 0.5, 1.0, 1.0, 0.5, 0.0, 0.5, -1.0]]]
    x = [[[1.0, -2.0, 3.0, 0.0, 2.0, -1.0, 4.0, 1.0, -3.0, 2.0, 1.0, -2.0],
          [2.0, 1.0, -1.0, 3.0, 0.0, -2.0, 1.0, 2.0, 0.0, -4.0, 3.0, 1.0]]]
    h0 = [[3.0, -2.0]]
    dh = [[[1.0, 0.0, -1.0, 2.0, 1.0, -2.0, 0.0, 1.0, 3.0, -1.0, 2.0, 1.0],
           [-1.0, 2.0, 1.0, 0.0, -2.0, 1.0, 3.0, -1.0, 0.0, 2.0, 1.0, -3.0]]]
    out = {"citation": "associative_scan_triton README: quick start, how it works",
           "layout": "dense [B=1, C=2, T=12]", "a": a, "x": x, "h0": h0, "dh": dh}
    for rev in (False, True):
        key = "reverse" if rev else "causal"
        h = oracle.scan_fwd(np.array(a), np.array(x), np.array(h0), reverse=rev)
        da, dx, dh0 = oracle.scan_bwd(np.array(a), np.array(x), np.array(dh), np.array(h0),
                                      reverse=rev)
        out[key] = {"h": h.tolist(), "da": da.tolist(), "dx": dx.tolist(), "dh0": dh0.tolist()}
    dump("scalar_dense_dyadic.json", out)


def scalar_packed():
    cu = [0, 3, 3, 7, 12]
    a = [[0.5, 1.0, 0.5, 0.0, -1.0, 0.5, 1.0, 0.5, 0.5, 1.0, -1.0, 0.5],
         [1.0, -1.0, 0.5, 0.5, 0.5, 0.0, 1.0, 1.0, 0.5, 0.0, 0.5, 1.0]]
    x = [[2.0, -1.0, 1.0, 3.0, 0.0, -2.0, 1.0, 4.0, -1.0, 2.0, 0.0, 1.0],
         [-1.0, 2.0, 0.0, 1.0, 3.0, -2.0, 2.0, 0.0, 1.0, -3.0, 2.0, -1.0]]
    h0 = [[1.0, -2.0], [5.0, 7.0], [-1.0, 2.0], [0.5, -0.5]]
    dh = [[1.0, -1.0, 2.0, 0.0, 1.0, 1.0, -2.0, 0.0, 3.0, 1.0, -1.0, 2.0],
          [0.0, 1.0, -1.0, 2.0, 1.0, 0.0, 1.0, -2.0, 1.0, 1.0, 0.0, -1.0]]
    out = {"citation": "associative_scan_triton README: quick start (cu_seqlens, "
                       "scan_bidirectional_branched), how it works",
           "layout": "packed [C=2, T=12], segment 1 is empty", "cu_seqlens": cu,
           "a": a, "x": x, "h0": h0, "dh": dh}
    for rev in (False, True):
        key = "reverse" if rev else "causal"
        h = oracle.scan_fwd(np.array(a), np.array(x), np.array(h0), cu_seqlens=np.array(cu),
                            reverse=rev)
        da, dx, dh0 = oracle.scan_bwd(np.array(a), np.array(x), np.array(dh), np.array(h0),
                                      cu_seqlens=np.array(cu), reverse=rev)
        out[key] = {"h": h.tolist(), "da": da.tolist(), "dx": dx.tolist(), "dh0": dh0.tolist()}
    dump("scalar_packed_dyadic.json", out)


def affine_2x2():
    rs = np.random.default_rng(1234)
    B, T, N, k, v = 1, 5, 2, 2, 2
    A = rs.choice([-1.0, -0.5, 0.0, 0.5, 1.0], size=(B, T, N, k, k))
    Bm = rs.integers(-3, 4, size=(B, T, N, k, v)).astype(np.float64)
    h0 = rs.integers(-2, 3, size=(B, N, k, v)).astype(np.float64)
    dH = rs.integers(-2, 3, size=(B, T, N, k, v)).astype(np.float64)
    H = oracle.affine_fwd(A, Bm, h0)
    dA, dB, dh0 = oracle.affine_bwd(A, Bm, dH, h0)
    dump("affine_2x2_dyadic.json", {
        "citation": "Triton scan kernels: One associative-scan family; Autograd integration "
                    "and the reversed-scan backward",
        "layout": "A [B=1,T=5,N=2,2,2], Bm/H [1,5,2,2,2], h0 [1,2,2,2]",
        "A": A.tolist(), "Bm": Bm.tolist(), "h0": h0.tolist(), "dH": dH.tolist(),
        "H": H.tolist(), "dA": dA.tolist(), "dB": dB.tolist(), "dh0": dh0.tolist()})


if __name__ == "__main__":
    scalar_dense()
    scalar_packed()
    affine_2x2()
