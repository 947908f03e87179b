"""Mamba-2 SSD forward scan for NVIDIA B300 (sm_103a).

Per head: h_t = exp(dt_t A) h_{t-1} + dt_t x_t B_t^T,  y_t = C_t^T h_t + D x_t.
``ssd_step_fwd`` is the same recurrence for one token per sequence (decoding);
``ssd_causal_conv1d_fwd`` and ``ssd_gated_rmsnorm_fwd`` are the block's steps before and after
the scan; ``ssd_scan_fwd_gated`` is the scan with the gated RMSNorm applied to its output.
The computation lives in ``libssd_scan.so`` (C ABI in ``include/ssd_scan.h``); this package is
its ctypes binding plus the seeded synthetic workloads (``workloads``).
"""
from ._binding import (  # noqa: F401
    LIB_PATH,
    PATH_NAMES,
    SSD_BF16,
    SSD_F32,
    SSD_PATH_AUTO,
    SSD_PATH_CHUNKED,
    SSD_PATH_TC,
    SSDError,
    load_library,
    ssd_causal_conv1d_fwd,
    ssd_gated_rmsnorm_fwd,
    make_dims,
    ssd_dims,
    ssd_scan_fwd,
    ssd_scan_fwd_gated,
    ssd_scan_fwd_host,
    ssd_scan_fwd_varlen,
    ssd_scan_gated_workspace_bytes,
    ssd_scan_get_status,
    ssd_scan_host_arena_bytes,
    ssd_scan_kernels_per_call,
    ssd_scan_resolve_path,
    ssd_scan_set_wait_cycles,
    ssd_block_get_status,
    ssd_scan_strerror,
    ssd_scan_varlen_workspace_bytes,
    ssd_scan_version,
    ssd_scan_workspace_bytes,
    ssd_step_fwd,
)
