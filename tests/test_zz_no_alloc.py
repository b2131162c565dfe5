"""scan_fwd_noalloc, the forward scan for callers that cannot allocate device
memory (memory-capped arenas, allocation-free real-time paths, plugin hosts
that only pass the tensors they own).

It is called through the C ABI and compared with scan_fwd on the same inputs
(same tolerance as the other parity tests), twice in a row, because every call
reuses the library's fixed scratch array. This file is collected last so that
a run stopping at the first failure has run every other test first; it also
passes alone in a fresh process.
"""

import pytest
import torch

from associative_affine_scan_gb300 import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
TOL = 1e-5


def rel_err(got, ref):
    d = (got.double() - ref.double()).abs() / ref.double().abs().clamp_min(1.0)
    return float(d.max()) if d.numel() else 0.0


def test_noalloc_matches_scan_fwd_dense_twice(lib):
    w = workloads.scalar_dense(2, 96, 3001, seed=31, h0=True)
    a, x, h0 = w.a.to(DEV), w.x.to(DEV), w.h0.to(DEV)
    out = torch.empty(a.shape, device=DEV)
    for rev in (False, True):
        ref = lib.scan_fwd(a, x, h0, None, rev)
        for _ in range(2):
            out.fill_(float("nan"))
            lib.scan_fwd_noalloc(a, x, h0, None, rev, out=out)
            torch.cuda.synchronize()
            assert rel_err(out, ref) <= TOL


def test_noalloc_matches_scan_fwd_packed_bf16_twice(lib):
    w = workloads.packed_bidir(seed=3, C=64, n_seqs=12, lo=1, hi=2000, p_reset=1e-3, h0=True)
    a, x, h0, cu = w.af.to(DEV), w.xf.to(DEV), w.h0f.to(DEV), w.cu_seqlens.to(DEV)
    for rev in (False, True):
        ref = lib.scan_fwd(a, x, h0, cu, rev)
        for _ in range(2):
            got = lib.scan_fwd_noalloc(a, x, h0, cu, rev)
            torch.cuda.synchronize()
            assert rel_err(got, ref) <= TOL


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    # 4096 rows x 2048 chunks of 512 steps need 128 MiB of summaries: the
    # host-side size check refuses before touching the (placeholder) pointers
    st = lib.lib().scan_fwd_noalloc(1024, 1024, None, None, 0, 1024, 1, 4096, 512 * 2048, 0, 0,
                                    None)
    assert st == lib.SCAN_ERR_WORKSPACE
