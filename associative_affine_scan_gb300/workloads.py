"""Seeded synthetic inputs for the scan, shared by the tests and the benchmark.

This module draws random numbers and lays them out; it holds none of the scan's
arithmetic. Everything is generated on the CPU with a seeded
``torch.Generator`` (one generator per call, tensors drawn in a fixed order), so
the CUDA path and the oracle see bit-identical inputs.

The named workloads follow the scalar benchmark shape of the
"associative_scan_triton" README (performance: B=8, C=1536, seqlen from 128 to
65536) and the block-matrix shape family of "Triton scan kernels" (Kernel
design: one (b, n) lane per state block, (k, v) blocks):

* ``single_sequence``  B=1, C=4, T=128, cu_seqlens=[0, 128], h0 = 0,
  a ~ U(0,1), x ~ N(0,1), dh ~ N(0,1)
* ``dense_4k``         [8, 1536, 4096] fp32, a ~ U(0,1), x ~ N(0,1),
  h0 ~ N(0,1), dh ~ N(0,1)
* ``dense_64k``        [8, 1536, 65536] fp32, a = sigmoid(z), z ~ N(2,1),
  x ~ N(0,1), h0 = 0, dh ~ N(0,1)
* ``packed_bidir``     C=2048, 64 sequences of length ~ U{512..8192} packed
  with int32 cu_seqlens, bf16 a ~ U(0,1) and x ~ N(0,1) per branch, resets
  (a = 0 at a packed position, all channels, both branches) with probability
  1e-3, fp32 dh ~ N(0,1) per branch
* ``affine_4x4``       B=8, T=4096, N=256, k=v=4, A = Q s with Q the
  orthogonal factor of a 4x4 N(0,1) matrix and s ~ U(0.9, 1.0) per matrix,
  B ~ N(0,1), h0 = 0, dH ~ N(0,1)
* ``log_4k``           [8, 1536, 4096] fp32, log a = logsigmoid(z),
  z ~ N(0,1), log x ~ N(0,1), no initial state, dh ~ N(0,1)
* ``rglru_4k``         [8, 1536, 4096] fp32 RG-LRU inputs ("Our RG-LRU GPU
  audit", Strengthened fused path): x, gate_a, gate_x ~ N(0,1), a_param ~
  U(4.3, 9) per channel (long memories: sigmoid(a_param)^8 from about 0.89 to
  0.999), segment_pos of documents with lengths ~ U{512..8192} laid end to end
  from t = 0 in every batch row, no initial state, dh ~ N(0,1)

Every generator takes a ``scale`` that shrinks the sizes for quick tests while
keeping the distributions.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


@dataclass
class ScalarWorkload:
    """Inputs of one scalar scan problem (dense [B,C,T] or packed [C,T])."""

    name: str
    a: torch.Tensor
    x: torch.Tensor
    dh: torch.Tensor
    h0: Optional[torch.Tensor] = None
    cu_seqlens: Optional[torch.Tensor] = None
    reverse: bool = False

    @property
    def n_elem(self) -> int:
        return self.a.numel()


@dataclass
class BidirWorkload:
    """Two independent branches over the same packed layout."""

    name: str
    af: torch.Tensor
    xf: torch.Tensor
    ar: torch.Tensor
    xr: torch.Tensor
    dhf: torch.Tensor
    dhr: torch.Tensor
    cu_seqlens: torch.Tensor
    resets: torch.Tensor = field(default=None)
    h0f: Optional[torch.Tensor] = None
    h0r: Optional[torch.Tensor] = None

    @property
    def n_elem(self) -> int:
        return self.af.numel() * 2


@dataclass
class AffineWorkload:
    name: str
    A: torch.Tensor
    Bm: torch.Tensor
    dH: torch.Tensor
    h0: Optional[torch.Tensor] = None

    @property
    def n_blocks(self) -> int:
        return self.A.shape[0] * self.A.shape[1] * self.A.shape[2]


@dataclass
class LogWorkload:
    name: str
    log_a: torch.Tensor
    log_x: torch.Tensor
    dh: torch.Tensor
    log_h0: Optional[torch.Tensor] = None
    cu_seqlens: Optional[torch.Tensor] = None

    @property
    def n_elem(self) -> int:
        return self.log_a.numel()


def scalar_dense(B: int, C: int, T: int, seed: int = 0, *, gate: str = "uniform",
                 h0: bool = True, dtype=torch.float32, name: str = "dense") -> ScalarWorkload:
    """Dense [B,C,T] inputs. gate: 'uniform' a~U(0,1); 'sigmoid2' a=sigmoid(N(2,1))."""
    g = _gen(seed)
    if gate == "uniform":
        a = torch.rand((B, C, T), generator=g)
    elif gate == "sigmoid2":
        a = torch.sigmoid(torch.randn((B, C, T), generator=g) + 2.0)
    else:
        raise ValueError(gate)
    x = torch.randn((B, C, T), generator=g)
    h0t = torch.randn((B, C), generator=g) if h0 else None
    dh = torch.randn((B, C, T), generator=g)
    return ScalarWorkload(name, a.to(dtype), x.to(dtype), dh, h0t)


def dense_beyond_int32(device, seed: int = 0) -> ScalarWorkload:
    """B=1, C=8200, T=262144 fp32 (2,149,580,800 elements, past 2^31): the
    dense recipe of dense_4k (a~U(0,1), x~N(0,1), h0~N(0,1), dh~N(0,1)),
    generated on `device` from a seeded generator of that device (34 GB of
    fp32 inputs; rows 8192.. start beyond element 2^31)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    shape = (1, 8200, 262144)
    a = torch.rand(shape, generator=g, device=device)
    x = torch.randn(shape, generator=g, device=device)
    h0t = torch.randn((1, 8200), generator=g, device=device)
    dh = torch.randn(shape, generator=g, device=device)
    return ScalarWorkload("dense_beyond_int32", a, x, dh, h0t)


def single_sequence(seed: int = 0) -> ScalarWorkload:
    g = _gen(seed)
    C, T = 4, 128
    a = torch.rand((C, T), generator=g)
    x = torch.randn((C, T), generator=g)
    dh = torch.randn((C, T), generator=g)
    cu = torch.tensor([0, T], dtype=torch.int32)
    return ScalarWorkload("single_sequence", a, x, dh, None, cu)


def dense_4k(seed: int = 0, scale: int = 1) -> ScalarWorkload:
    return scalar_dense(8, 1536 // scale, 4096, seed, gate="uniform", h0=True, name="dense_4k")


def dense_64k(seed: int = 0, scale: int = 1) -> ScalarWorkload:
    return scalar_dense(8, 1536 // scale, 65536, seed, gate="sigmoid2", h0=False, name="dense_64k")


def packed_lengths(n_seqs: int, lo: int, hi: int, g: torch.Generator) -> torch.Tensor:
    """Integer lengths ~ U{lo..hi} (inclusive) and their exclusive cumsum."""
    lens = torch.randint(lo, hi + 1, (n_seqs,), generator=g, dtype=torch.int64)
    cu = torch.zeros(n_seqs + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lens, 0)
    return cu.to(torch.int32)


def packed_bidir(seed: int = 0, C: int = 2048, n_seqs: int = 64, lo: int = 512, hi: int = 8192,
                 p_reset: float = 1e-3, dtype=torch.bfloat16, h0: bool = False,
                 name: str = "packed_bidir") -> BidirWorkload:
    g = _gen(seed)
    cu = packed_lengths(n_seqs, lo, hi, g)
    T = int(cu[-1])
    resets = torch.rand((T,), generator=g) < p_reset
    keep = (~resets).to(torch.float32)

    def gate():
        return (torch.rand((C, T), generator=g) * keep).to(dtype)

    af = gate()
    xf = torch.randn((C, T), generator=g).to(dtype)
    ar = gate()
    xr = torch.randn((C, T), generator=g).to(dtype)
    dhf = torch.randn((C, T), generator=g)
    dhr = torch.randn((C, T), generator=g)
    h0f = torch.randn((n_seqs, C), generator=g) if h0 else None
    h0r = torch.randn((n_seqs, C), generator=g) if h0 else None
    return BidirWorkload(name, af, xf, ar, xr, dhf, dhr, cu, resets, h0f, h0r)


def _orthogonal_4x4(n: int, k: int, g: torch.Generator) -> torch.Tensor:
    """Orthogonal factors of n random N(0,1) k x k matrices (Gram-Schmidt on columns)."""
    M = torch.randn((n, k, k), generator=g, dtype=torch.float64)
    Q = torch.empty_like(M)
    for j in range(k):
        v = M[:, :, j].clone()
        for i in range(j):
            v -= (Q[:, :, i] * M[:, :, j]).sum(-1, keepdim=True) * Q[:, :, i]
        Q[:, :, j] = v / v.norm(dim=-1, keepdim=True)
    return Q


def affine(B: int, T: int, N: int, k: int, v: int, seed: int = 0, *, h0: bool = False,
           name: str = "affine") -> AffineWorkload:
    g = _gen(seed)
    Q = _orthogonal_4x4(B * T * N, k, g)
    s = torch.rand((B * T * N, 1, 1), generator=g, dtype=torch.float64) * 0.1 + 0.9
    A = (Q * s).to(torch.float32).reshape(B, T, N, k, k)
    Bm = torch.randn((B, T, N, k, v), generator=g)
    dH = torch.randn((B, T, N, k, v), generator=g)
    h0t = torch.randn((B, N, k, v), generator=g) if h0 else None
    return AffineWorkload(name, A, Bm, dH, h0t)


def affine_4x4(seed: int = 0, scale: int = 1) -> AffineWorkload:
    return affine(8, 4096 // scale, 256, 4, 4, seed, name="affine_4x4")


@dataclass
class GdnWorkload:
    name: str
    alpha: torch.Tensor  # [B,H,T]
    b: torch.Tensor      # [B,H,T,S]
    v: torch.Tensor      # [B,H,T,D]
    c: torch.Tensor      # [B,H,T,S]
    dout: torch.Tensor   # [B,H,T,D]
    h0: Optional[torch.Tensor] = None  # [B,H,S,D]

    @property
    def n_steps(self) -> int:
        return self.alpha.numel()


def gdn(B: int, H: int, T: int, S: int, D: int, seed: int = 0, *, h0: bool = False,
        name: str = "gdn") -> GdnWorkload:
    """Scalar-gated outer-product state inputs: gates alpha = sigmoid(z),
    z~N(3,1) (decays near 1), keys b, c ~ N(0,1)/sqrt(S), values v ~ N(0,1),
    upstream gradient dout ~ N(0,1), optional h0 ~ N(0,1); fp32, drawn in
    that order from one CPU generator."""
    g = _gen(seed)
    alpha = torch.sigmoid(torch.randn((B, H, T), generator=g) + 3.0)
    b = torch.randn((B, H, T, S), generator=g) / S ** 0.5
    v = torch.randn((B, H, T, D), generator=g)
    c = torch.randn((B, H, T, S), generator=g) / S ** 0.5
    dout = torch.randn((B, H, T, D), generator=g)
    h0t = torch.randn((B, H, S, D), generator=g) if h0 else None
    return GdnWorkload(name, alpha, b, v, c, dout, h0t)


def gdn_4k(seed: int = 0) -> GdnWorkload:
    """8 batches x 32 heads x 4096 steps, (S, D) = (32, 32): the state shape
    and chunked T of the GDN page's worked setting."""
    return gdn(8, 32, 4096, 32, 32, seed, name="gdn_4k")


def log_dense(B: int, C: int, T: int, seed: int = 0, *, h0: bool = False,
              name: str = "log") -> LogWorkload:
    g = _gen(seed)
    log_a = torch.nn.functional.logsigmoid(torch.randn((B, C, T), generator=g))
    log_x = torch.randn((B, C, T), generator=g)
    dh = torch.randn((B, C, T), generator=g)
    lh0 = torch.randn((B, C), generator=g) if h0 else None
    return LogWorkload(name, log_a, log_x, dh, lh0)


def log_4k(seed: int = 0, scale: int = 1) -> LogWorkload:
    return log_dense(8, 1536 // scale, 4096, seed, name="log_4k")


@dataclass
class RglruWorkload:
    """Inputs of one RG-LRU problem: x, gate logits [B, C, T], a_param [C],
    segment_pos int32 [B, T] (or None), h0 [B, C] (or None), dh [B, C, T]."""

    name: str
    x: torch.Tensor
    gate_a: torch.Tensor
    gate_x: torch.Tensor
    a_param: torch.Tensor
    dh: torch.Tensor
    segment_pos: Optional[torch.Tensor] = None
    h0: Optional[torch.Tensor] = None

    @property
    def n_elem(self) -> int:
        return self.x.numel()


def document_positions(B: int, T: int, lo: int, hi: int, g: torch.Generator) -> torch.Tensor:
    """segment_pos [B, T]: per batch row, documents of lengths ~ U{lo..hi} laid
    end to end from t = 0; the value is the step's position in its document."""
    pos = torch.empty((B, T), dtype=torch.int32)
    for b in range(B):
        t = 0
        while t < T:
            n = int(torch.randint(lo, hi + 1, (1,), generator=g))
            m = min(n, T - t)
            pos[b, t:t + m] = torch.arange(m, dtype=torch.int32)
            t += m
    return pos


def rglru(B: int, C: int, T: int, seed: int = 0, *, docs: Optional[tuple] = (512, 8192),
          h0: bool = False, dtype=torch.float32, name: str = "rglru") -> RglruWorkload:
    """x, gate_a, gate_x ~ N(0,1) (stored in `dtype`); a_param ~ U(4.3, 9);
    segment_pos of documents with lengths ~ U{docs} (None: no resets);
    dh ~ N(0,1); h0 ~ N(0,1) if asked. Drawn in that order from one generator."""
    g = _gen(seed)
    x = torch.randn((B, C, T), generator=g).to(dtype)
    ga = torch.randn((B, C, T), generator=g).to(dtype)
    gx = torch.randn((B, C, T), generator=g).to(dtype)
    ap = 4.3 + 4.7 * torch.rand((C,), generator=g)
    seg = document_positions(B, T, docs[0], docs[1], g) if docs else None
    dh = torch.randn((B, C, T), generator=g)
    h0t = torch.randn((B, C), generator=g) if h0 else None
    return RglruWorkload(name, x, ga, gx, ap, dh, seg, h0t)


def rglru_4k(seed: int = 0) -> RglruWorkload:
    """8 x 1536 x 4096, the scalar benchmark's dense shape, with documents of
    the packed benchmark's length mix."""
    return rglru(8, 1536, 4096, seed, name="rglru_4k")
