"""scan_fwd_noalloc, the forward scan for callers that cannot allocate device
memory (memory-capped arenas, allocation-free real-time paths, plugin hosts
that only pass the tensors they own).

It is called through the C ABI and compared with scan_fwd on the same inputs
and with the fp64 oracle (1e-5 of max(1, |ref|) for its fp32 output), twice
in a row, because every call reuses the library's fixed scratch array. The
cases cover short rows (T <= 256: one- and two-block chunks), row counts that
leave a partial group of 4 rows, no initial state, fp32 and bf16 packed rows,
more sequences than the shared-memory offset table holds (4096 entries), the
first call of the file made on a side stream, guard bands around the output,
and the read-back of a finding of the kernel's own checks. This file is collected last so that a run stopping at the first
failure has run every other test first; it also passes alone in a fresh
process.
"""

import numpy as np
import pytest
import torch

import oracle
from associative_affine_scan_gb300 import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
TOL = 1e-5
PAD = 1024
SENTINEL = 0x7FC0DEAD


def rel_err(got, ref):
    got = got.detach().double().cpu().numpy()
    ref = np.asarray(ref.detach().double().cpu().numpy() if hasattr(ref, "detach") else ref,
                     dtype=np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref))))


def check_twice(lib, a, x, h0, cu, rev, stream=None, out=None):
    """Two calls in a row against scan_fwd and the oracle."""
    ref = lib.scan_fwd(a, x, h0, cu, rev)
    gold = oracle.scan_fwd(a.cpu(), x.cpu(), None if h0 is None else h0.cpu(),
                           None if cu is None else cu.cpu(), rev)
    for _ in range(2):
        got = lib.scan_fwd_noalloc(a, x, h0, cu, rev, out=out, stream=stream)
        if stream is not None:
            stream.synchronize()
        torch.cuda.synchronize()
        assert rel_err(got, ref) <= TOL
        assert rel_err(got, gold) <= TOL


def packed(C, lens, seed, dtype, h0=True):
    g = torch.Generator().manual_seed(seed)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    T = int(cu[-1])
    a = torch.rand((C, T), generator=g)
    a[:, torch.rand(T, generator=g) < 1e-3] = 0.0
    x = torch.randn((C, T), generator=g)
    hz = torch.randn((len(lens), C), generator=g) if h0 else None
    return (a.to(dtype).to(DEV), x.to(dtype).to(DEV), None if hz is None else hz.to(DEV),
            cu.to(DEV))


def test_noalloc_first_call_on_a_side_stream(lib):
    """The file's first call runs on a torch side stream (non-blocking with
    respect to the legacy default stream): its set-up queues nothing, so the
    kernel on that stream starts from the scratch as the module load left it."""
    w = workloads.scalar_dense(2, 96, 3001, seed=30, h0=True)
    a, x, h0 = w.a.to(DEV), w.x.to(DEV), w.h0.to(DEV)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    out = torch.empty(a.shape, device=DEV)
    for rev in (False, True):
        check_twice(lib, a, x, h0, None, rev, stream=side, out=out)


@pytest.mark.parametrize("B,C,T", [(2, 96, 3001), (1, 7, 1), (1, 7, 100), (3, 5, 256),
                                   (2, 3, 257), (1, 1, 5000), (1, 2, 4100)])
@pytest.mark.parametrize("with_h0", [True, False])
def test_noalloc_dense_twice(lib, B, C, T, with_h0):
    w = workloads.scalar_dense(B, C, T, seed=B * 1000 + C + T, h0=True)
    a, x = w.a.to(DEV), w.x.to(DEV)
    h0 = w.h0.to(DEV) if with_h0 else None
    for rev in (False, True):
        check_twice(lib, a, x, h0, None, rev)


def test_noalloc_dense_bf16_twice(lib):
    w = workloads.scalar_dense(2, 33, 2049, seed=8, h0=True, dtype=torch.bfloat16)
    a, x, h0 = w.a.to(DEV), w.x.to(DEV), w.h0.to(DEV)
    for rev in (False, True):
        check_twice(lib, a, x, h0, None, rev)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("with_h0", [True, False])
def test_noalloc_packed_twice(lib, dtype, with_h0):
    w = workloads.packed_bidir(seed=3, C=64, n_seqs=12, lo=1, hi=2000, p_reset=1e-3,
                               dtype=dtype, h0=True)
    a, x, cu = w.af.to(DEV), w.xf.to(DEV), w.cu_seqlens.to(DEV)
    h0 = w.h0f.to(DEV) if with_h0 else None
    for rev in (False, True):
        check_twice(lib, a, x, h0, cu, rev)


def test_noalloc_more_sequences_than_the_offset_table(lib):
    """5000 packed sequences (lengths 0..40): the offsets stay in global
    memory, as in scan_fwd."""
    g = np.random.default_rng(12)
    lens = g.integers(0, 41, size=5000).tolist()
    a, x, h0, cu = packed(6, lens, seed=13, dtype=torch.float32)
    for rev in (False, True):
        check_twice(lib, a, x, h0, cu, rev)


@pytest.mark.parametrize("shift", [0, 1])
def test_noalloc_guard_bands(lib, shift):
    """The output inside a sentinel-filled buffer: nothing written outside it,
    every element inside written."""
    for T in (1, 3, 129, 4097):
        w = workloads.scalar_dense(2, 5, T, seed=T + 1, h0=True)
        a, x, h0 = w.a.to(DEV), w.x.to(DEV), w.h0.to(DEV)
        n = a.numel()
        buf = torch.empty(n + 2 * PAD + shift, dtype=torch.float32, device=DEV)
        bits = buf.view(torch.int32)
        bits.fill_(SENTINEL)
        lo = PAD + shift
        out = buf[lo:lo + n].view(a.shape)
        for rev in (False, True):
            lib.scan_fwd_noalloc(a, x, h0, None, rev, out=out)
            torch.cuda.synchronize()
            assert bool((bits[:lo] == SENTINEL).all()) and bool((bits[lo + n:] == SENTINEL).all())
            assert rel_err(out, oracle.scan_fwd(w.a, w.x, w.h0, None, rev)) <= TOL


def test_noalloc_device_status_reads_back_and_clears(lib):
    """A device cu_seqlens that is not non-decreasing (every entry still in
    [0, T], so every sequence index the kernel forms stays in 0 .. n - 1)
    returns SCAN_OK from the host checks; the kernel's own check records
    SCAN_ERR_SEQLENS in the library's scratch, which the accessor reads once
    and clears. Calls before and after still match the oracle."""
    a, x, h0, cu = packed(4, [100, 200], seed=31, dtype=torch.float32)
    check_twice(lib, a, x, h0, cu, False)
    assert lib.scan_noalloc_device_status(DEV) == lib.SCAN_OK
    bad = torch.tensor([0, 200, 100, 300], dtype=torch.int32, device=DEV)
    h0b = torch.zeros(3, 4, device=DEV)
    lib.scan_fwd_noalloc(a, x, h0b, bad)
    assert lib.scan_noalloc_device_status(DEV) == lib.SCAN_ERR_SEQLENS
    assert lib.scan_noalloc_device_status(DEV) == lib.SCAN_OK
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    lib.scan_fwd_noalloc(a, x, h0b, bad, True, stream=side)
    assert lib.scan_noalloc_device_status(DEV, stream=side) == lib.SCAN_ERR_SEQLENS
    check_twice(lib, a, x, h0, cu, True)
    assert lib.scan_noalloc_device_status(DEV) == lib.SCAN_OK


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    # 4096 rows x 2048 chunks of 512 steps need 128 MiB of summaries: the
    # host-side size check refuses before touching the (placeholder) pointers
    st = lib.lib().scan_fwd_noalloc(1024, 1024, None, None, 0, 1024, 1, 4096, 512 * 2048, 0, 0,
                                    None)
    assert st == lib.SCAN_ERR_WORKSPACE


def test_noalloc_rejects_host_pointers(lib):
    """The tensors must be on the current device: host memory is refused."""
    a = torch.rand(1, 2, 64)
    st = lib.lib().scan_fwd_noalloc(a.data_ptr(), a.data_ptr(), None, None, 0, a.data_ptr(), 1, 2,
                                    64, 0, 0, None)
    assert st == lib.SCAN_ERR_INVALID_ARG
