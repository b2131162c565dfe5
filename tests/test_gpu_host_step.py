"""scan_step_host: the scan and its backward on dense rows in host memory,
pipelined over row pieces ("Triton scan kernels": the forward scan and the
reversed-scan backward; the dense rows are independent recurrences). Its
results must equal those of scan_fwd and scan_bwd run on the device buffers
with the same variant: the same kernels on the same rows, bit for bit when T
is a multiple of 4. Otherwise a piece's first row starts at another 4-element
memory phase, which moves the kernels' run boundaries (and so the rounding):
then fp32 results agree within 1e-5 (of max(1, |ref|)) and bf16 ones within
1e-2. The host results are also compared with the fp64 oracle: every row of
the small cases, 64 rows (the first, the last and 62 drawn at random) of the
8 x 1536 x 4096 one."""

import numpy as np
import pytest
import torch

import oracle
from associative_affine_scan_gb300 import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _host_step(lib, w, pieces, with_h0, dtype):
    a, x, dh = (t.to(dtype) if t is not w.dh else t for t in (w.a, w.x, w.dh))
    h0 = w.h0 if with_h0 else None
    pin = lambda t: None if t is None else t.contiguous().pin_memory()
    ha, hx, hdh, hh0 = pin(a), pin(x), pin(dh), pin(h0)
    B, C, T = a.shape
    out = (torch.empty(B, C, T).pin_memory(), torch.empty(B, C, T, dtype=dtype).pin_memory(),
           torch.empty(B, C, T, dtype=dtype).pin_memory(),
           torch.empty(B, C).pin_memory() if with_h0 else None)
    dev = (torch.empty(B, C, T, dtype=dtype, device=DEV), torch.empty(B, C, T, dtype=dtype, device=DEV),
           torch.empty(B, C, device=DEV) if with_h0 else None, torch.empty(B, C, T, device=DEV),
           torch.empty(B, C, T, device=DEV), torch.empty(B, C, T, dtype=dtype, device=DEV),
           torch.empty(B, C, T, dtype=dtype, device=DEV),
           torch.empty(B, C, device=DEV) if with_h0 else None)
    lib.scan_step_host(ha, hx, hdh, hh0, out=out, device=dev, pieces=pieces)
    torch.cuda.synchronize()
    # reference: the same calls on device copies, stationary variant
    o = lib.ScanOpts()
    o.variant = lib.SCAN_VARIANT_STATIONARY
    da_, xa_, dha = a.to(DEV), x.to(DEV), dh.to(DEV)
    h0a = h0.to(DEV) if with_h0 else None
    h = lib.scan_fwd(da_, xa_, h0a, opts=o)
    gda, gdx, gdh0 = lib.scan_bwd(da_, h, dha, h0a, opts=o)
    torch.cuda.synchronize()
    pairs = [(out[0], h), (out[1], gda), (out[2], gdx)] + ([(out[3], gdh0)] if with_h0 else [])
    for got, ref in pairs:
        ref = ref.cpu()
        if T % 4 == 0:
            assert torch.equal(got, ref)
        else:
            tol = 1e-5 if got.dtype == torch.float32 else 1e-2
            g, r = got.double(), ref.double()
            assert ((g - r).abs() / r.abs().clamp(min=1.0)).max().item() <= tol
    _against_oracle(a, x, dh, h0, out)


def _against_oracle(a, x, dh, h0, out):
    """Host results of the step against the fp64 oracle on the same inputs
    (bf16 inputs are read exactly): h, dh0 within 1e-5, da, dx within 1e-5
    (fp32) or 1e-2 (stored in bf16)."""
    B, C, T = a.shape
    rows = B * C
    if rows * T <= (1 << 21):
        pick = np.arange(rows)
    else:
        g = np.random.default_rng(7)
        pick = np.unique(np.concatenate([[0, rows - 1], g.choice(rows, 62, replace=False)]))
    sel = lambda t: t.reshape(rows, -1)[torch.from_numpy(pick)][None]
    r_h = oracle.scan_fwd(sel(a), sel(x), None if h0 is None else sel(h0)[..., 0])
    r_da, r_dx, r_dh0 = oracle.scan_bwd(sel(a), sel(x), sel(dh),
                                        None if h0 is None else sel(h0)[..., 0])
    tol_g = 1e-5 if a.dtype == torch.float32 else 1e-2

    def err(got, ref):
        got = got.double().numpy()
        return float(np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref))))

    assert err(sel(out[0]), r_h) <= 1e-5
    assert err(sel(out[1]), r_da) <= tol_g
    assert err(sel(out[2]), r_dx) <= tol_g
    if h0 is not None:
        assert err(sel(out[3])[..., 0], r_dh0) <= 1e-5


@pytest.mark.parametrize("pieces", [0, 1, 3, 7, 64])
@pytest.mark.parametrize("with_h0", [True, False])
def test_host_step_equals_device_calls_f32(lib, pieces, with_h0):
    w = workloads.scalar_dense(3, 37, 1000, seed=21 + pieces, h0=True)
    _host_step(lib, w, pieces, with_h0, torch.float32)


@pytest.mark.parametrize("T", [768, 777])
def test_host_step_bf16_inputs(lib, T):
    w = workloads.scalar_dense(2, 64, T, seed=5, h0=True)
    _host_step(lib, w, 5, True, torch.bfloat16)


def test_host_step_ragged_t_f32(lib):
    w = workloads.scalar_dense(2, 45, 1001, seed=9, h0=True)
    _host_step(lib, w, 4, True, torch.float32)


def test_host_step_dense_4k_sample_pieces(lib):
    """The bench's e2e configuration (8 x 1536 x 4096, 8 pieces)."""
    w = workloads.dense_4k(seed=0)
    _host_step(lib, w, 0, w.h0 is not None, torch.float32)
