"""The seeded synthetic inputs follow the recipes the design notes state for
each workload (shapes, dtypes, value ranges, the packed config's sequence
lengths and shared resets, the RG-LRU documents), and the same seed gives the
same tensors. CPU only; the full-size workloads are checked at reduced channel
counts where their recipe does not depend on the channel count."""

import math

import torch

from associative_affine_scan_gb300 import workloads


def test_same_seed_same_inputs_other_seed_other_inputs():
    w0, w1, w2 = (workloads.dense_4k(seed=s, scale=256) for s in (0, 0, 1))
    for name in ("a", "x", "dh", "h0"):
        assert torch.equal(getattr(w0, name), getattr(w1, name))
        assert not torch.equal(getattr(w0, name), getattr(w2, name))


def test_dense_recipes():
    w = workloads.dense_4k(seed=0, scale=64)  # 8 x 24 x 4096
    assert w.a.shape == (8, 24, 4096) and w.a.dtype == torch.float32
    assert w.h0.shape == (8, 24) and w.cu_seqlens is None
    assert float(w.a.min()) >= 0.0 and float(w.a.max()) < 1.0  # a ~ U(0, 1)
    assert abs(float(w.a.mean()) - 0.5) < 0.01
    assert abs(float(w.x.std()) - 1.0) < 0.01 and abs(float(w.dh.std()) - 1.0) < 0.01
    w = workloads.dense_64k(seed=0, scale=1536)  # 8 x 1 x 65536
    assert w.a.shape == (8, 1, 65536) and w.h0 is None
    z = torch.logit(w.a.double())  # a = sigmoid(z), z ~ N(2, 1)
    assert abs(float(z.mean()) - 2.0) < 0.02 and abs(float(z.std()) - 1.0) < 0.02
    w = workloads.single_sequence(seed=0)
    assert w.a.shape == (4, 128) and w.cu_seqlens.tolist() == [0, 128] and w.h0 is None


def test_packed_bidir_lengths_and_shared_resets():
    """64 sequences of lengths U{512..8192}; the lengths and resets are drawn
    first, so a 4-channel draw has the full config's: sum of lengths 275,479
    for seed 0. Resets (a = 0 exactly) at Bernoulli(1e-3) packed positions,
    shared by every channel and both branches."""
    w = workloads.packed_bidir(seed=0, C=4)
    cu = w.cu_seqlens
    lens = (cu[1:] - cu[:-1]).tolist()
    assert len(lens) == 64 and cu[0] == 0 and int(cu[-1]) == 275479
    assert min(lens) >= 512 and max(lens) <= 8192
    T = int(cu[-1])
    n_reset = int(w.resets.sum())
    assert abs(n_reset - 1e-3 * T) < 4 * math.sqrt(1e-3 * T)
    for a in (w.af, w.ar):
        assert a.dtype == torch.bfloat16 and a.shape == (4, T)
        assert bool((a[:, w.resets] == 0).all())
        assert int((a == 0).sum()) == 4 * n_reset  # U(0,1) gives no other exact zero here
    assert w.dhf.dtype == torch.float32 and w.h0f is None


def test_affine_gates_are_scaled_orthogonal():
    """A = Q s, Q orthogonal (Gram-Schmidt of an N(0,1) matrix), s ~ U(0.9, 1):
    A^T A = s^2 I."""
    w = workloads.affine(2, 16, 3, 4, 4, seed=0, h0=True)
    A = w.A.double()
    AtA = A.transpose(-1, -2) @ A
    s2 = AtA.diagonal(dim1=-2, dim2=-1).mean(-1)
    assert float((AtA - s2[..., None, None] * torch.eye(4, dtype=torch.float64)).abs().max()) < 1e-6
    s = s2.sqrt()
    assert float(s.min()) >= 0.9 - 1e-6 and float(s.max()) <= 1.0 + 1e-6
    assert w.Bm.shape == (2, 16, 3, 4, 4) and w.h0.shape == (2, 3, 4, 4)


def test_gdn_recipe():
    w = workloads.gdn(4, 8, 512, 32, 16, seed=0, h0=True)
    assert w.alpha.shape == (4, 8, 512) and w.b.shape == (4, 8, 512, 32)
    assert w.v.shape == (4, 8, 512, 16) and w.h0.shape == (4, 8, 32, 16)
    z = torch.logit(w.alpha.double())  # alpha = sigmoid(z), z ~ N(3, 1)
    assert abs(float(z.mean()) - 3.0) < 0.02 and abs(float(z.std()) - 1.0) < 0.02
    assert abs(float(w.b.std()) * math.sqrt(32) - 1.0) < 0.01  # keys ~ N(0, 1) / sqrt(S)
    assert abs(float(w.c.std()) * math.sqrt(32) - 1.0) < 0.01
    assert abs(float(w.v.std()) - 1.0) < 0.01


def test_rglru_recipe_and_documents():
    """a_param ~ U(4.3, 9); segment_pos counts the steps of documents of
    lengths U{512..8192} laid end to end from t = 0 in every batch row (the
    last one cut at T)."""
    B, C, T = 3, 64, 20000
    w = workloads.rglru(B, C, T, seed=0)
    assert float(w.a_param.min()) >= 4.3 and float(w.a_param.max()) <= 9.0
    seg = w.segment_pos
    assert seg.shape == (B, T) and seg.dtype == torch.int32
    for b in range(B):
        row = seg[b]
        assert int(row[0]) == 0
        starts = (row == 0).nonzero().flatten().tolist() + [T]
        for s, e in zip(starts[:-1], starts[1:]):
            assert torch.equal(row[s:e], torch.arange(e - s, dtype=torch.int32))
            if e < T:
                assert 512 <= e - s <= 8192
    w16 = workloads.rglru(2, 4, 100, seed=1, docs=None, dtype=torch.bfloat16, h0=True)
    assert w16.segment_pos is None and w16.x.dtype == torch.bfloat16 and w16.h0.shape == (2, 4)
    assert w16.dh.dtype == torch.float32
