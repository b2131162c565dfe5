"""The Python binding fails loudly instead of computing anywhere but the GPU:
CPU tensors are refused before any library call, and a missing libscan.so
raises on first use. CPU only."""

import pytest
import torch

import associative_affine_scan_gb300 as scan
from associative_affine_scan_gb300 import _binding


def _cpu(*shape, dtype=torch.float32):
    return torch.zeros(shape, dtype=dtype)


@pytest.mark.parametrize("call", [
    lambda: scan.scan_fwd(_cpu(1, 2, 8), _cpu(1, 2, 8)),
    lambda: scan.scan_bwd(_cpu(1, 2, 8), _cpu(1, 2, 8), _cpu(1, 2, 8)),
    lambda: scan.scan_bidir_fwd(_cpu(2, 8), _cpu(2, 8), _cpu(2, 8), _cpu(2, 8), None, None,
                                torch.tensor([0, 8], dtype=torch.int32)),
    lambda: scan.scan_log_fwd(_cpu(1, 2, 8), _cpu(1, 2, 8)),
    lambda: scan.affine_scan_fwd(_cpu(1, 8, 2, 4, 4), _cpu(1, 8, 2, 4, 4)),
    lambda: scan.affine_prefix_fwd(_cpu(1, 8, 2, 4, 4)),
    lambda: scan.gdn_fwd(_cpu(1, 2, 8), _cpu(1, 2, 8, 16), _cpu(1, 2, 8, 16), _cpu(1, 2, 8, 16)),
    lambda: scan.scan_fwd_noalloc(_cpu(1, 2, 8), _cpu(1, 2, 8)),
    lambda: scan.scan_bidir_bwd(_cpu(2, 8), _cpu(2, 8), _cpu(2, 8), _cpu(2, 8), _cpu(2, 8),
                                _cpu(2, 8), None, None, torch.tensor([0, 8], dtype=torch.int32)),
    lambda: scan.scan_log_bwd(_cpu(1, 2, 8), _cpu(1, 2, 8), _cpu(1, 2, 8), _cpu(1, 2, 8)),
    lambda: scan.affine_scan_bwd(_cpu(1, 8, 2, 4, 4), _cpu(1, 8, 2, 4, 4), _cpu(1, 8, 2, 4, 4)),
    lambda: scan.affine_prefix_bwd(_cpu(1, 8, 2, 4, 4), _cpu(1, 8, 2, 4, 4), _cpu(1, 8, 2, 4, 4)),
    lambda: scan.gdn_bwd(_cpu(1, 2, 8), _cpu(1, 2, 8, 16), _cpu(1, 2, 8, 16), _cpu(1, 2, 8, 16),
                         _cpu(256), _cpu(1, 2, 8, 16)),
    lambda: scan.rglru_fwd(_cpu(1, 2, 8), _cpu(1, 2, 8), _cpu(1, 2, 8), _cpu(2)),
    lambda: scan.rglru_bwd(_cpu(1, 2, 8), _cpu(1, 2, 8), _cpu(1, 2, 8), _cpu(2), _cpu(1, 2, 8),
                           _cpu(1, 2, 8)),
    lambda: scan.scan_copy(_cpu(1024), _cpu(1024)),
])
def test_cpu_tensors_are_refused(call):
    with pytest.raises(ValueError, match="CUDA tensor"):
        call()


def test_non_tensors_are_refused():
    with pytest.raises(TypeError, match="torch.Tensor"):
        scan.scan_fwd([0.0] * 8, [0.0] * 8)


def test_missing_library_raises(monkeypatch):
    monkeypatch.setattr(_binding, "_lib_handle", None)
    monkeypatch.setattr(_binding, "LIB_PATH", _binding.LIB_PATH + ".absent")
    with pytest.raises(ImportError, match="missing"):
        _binding.lib()


def test_unknown_options_are_refused():
    """A misspelt option name raises instead of leaving the planner's choice
    in place; the known names set the structure's fields."""
    with pytest.raises(ValueError, match="unknown scan option 'chunks'"):
        _binding._opts({"chunks": 256})
    o = _binding._opts({"chunk": 256, "rows_per_cta": 2, "variant": scan.SCAN_VARIANT_LOOKBACK,
                        "wait_limit_s": 0.5, "cu_seqlens_host": [0, 3, 8]})
    assert (o.chunk, o.rows_per_cta, o.variant, o.wait_limit_s) == (256, 2, scan.SCAN_VARIANT_LOOKBACK, 0.5)
    assert [o.cu_seqlens_host[i] for i in range(3)] == [0, 3, 8]
