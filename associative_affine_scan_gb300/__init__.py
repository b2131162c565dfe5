"""libscan: the associative affine scan h_t = A_t h_{t-1} + B_t on one GB300.

The compute lives in ``libscan.so`` (hand-written CUDA for sm_103a behind the
C ABI in ``include/libscan.h``); this package is its thin ctypes binding, with
one Python function per C entry point and the same names. Importing the package
does not load the library; the first call does, and fails loudly if it is
missing (there is no CPU fallback).

``workloads`` holds the seeded synthetic inputs used by the tests and the
benchmark.
"""

from ._binding import (  # noqa: F401
    EXPORTED,
    LIB_PATH,
    SCAN_BF16,
    SCAN_COPY_TMA,
    SCAN_COPY_VEC,
    SCAN_ERR_ALIGNMENT,
    SCAN_ERR_CUDA,
    SCAN_ERR_INVALID_ARG,
    SCAN_ERR_SEQLENS,
    SCAN_ERR_TIMEOUT,
    SCAN_ERR_UNSUPPORTED,
    SCAN_ERR_WORKSPACE,
    SCAN_F32,
    SCAN_OK,
    SCAN_OP_AFFINE_BWD,
    SCAN_OP_AFFINE_FWD,
    SCAN_OP_BIDIR_BWD,
    SCAN_OP_BIDIR_FWD,
    SCAN_OP_BWD,
    SCAN_OP_FWD,
    SCAN_OP_LOG_BWD,
    SCAN_OP_LOG_FWD,
    SCAN_VARIANT_AUTO,
    SCAN_VARIANT_LOOKBACK,
    SCAN_VARIANT_STREAM,
    SCAN_VARIANT_STATIONARY,
    ScanError,
    ScanOpts,
    affine_scan_bwd,
    affine_prefix_fwd,
    affine_prefix_bwd,
    gdn_checkpoint_bytes,
    gdn_fwd,
    gdn_workspace_bytes,
    gdn_bwd,
    affine_scan_fwd,
    lib,
    rglru_bwd,
    rglru_fwd,
    scan_bidir_bwd,
    scan_bidir_fwd,
    scan_bwd,
    scan_copy,
    scan_fwd,
    scan_fwd_noalloc,
    scan_noalloc_device_status,
    scan_step_host,
    scan_get_device_status,
    scan_log_fwd,
    scan_log_bwd,
    scan_status_string,
    scan_version,
    scan_workspace_bytes,
    scan_workspace_init,
)
