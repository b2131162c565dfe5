"""Shared pytest setup: the ``gpu`` marker and the repository root on sys.path."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libscan")


def cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover - torch missing
        return False


@pytest.fixture(scope="session")
def lib():
    """The CUDA binding; a GPU test that cannot get it fails loudly."""
    if not cuda_available():
        pytest.fail("gpu test selected but no CUDA device is visible")
    import associative_affine_scan_gb300 as scan
    return scan
