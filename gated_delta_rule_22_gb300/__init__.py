"""Gated delta rule training kernels for NVIDIA GB300 (sm_103a).

The compute lives in libgdn.so, a C-ABI library of hand-written CUDA kernels
(include/gdn.h). This package is its thin Python binding.
"""
from .binding import (  # noqa: F401
    GDN_BF16, GDN_F32, GdnError, GdnShape, gdn_bwd, gdn_bwd_noalloc, gdn_bwd_workspace_bytes,
    gdn_ckpt_bytes, gdn_debug_wait_probe, gdn_device_status, gdn_diag_fma_tflops, gdn_fwd,
    gdn_bwd_seg, gdn_fwd_seg, gdn_gates_bwd, gdn_gates_fwd, gdn_last_error, gdn_seg_ckpt_bytes,
    gdn_seg_workspace_bytes, gdn_seg_choose, gdn_fwd_infer, gdn_infer_workspace_bytes, gdn_bwd_rc, gdn_fwd_rc, gdn_rc_bwd_workspace_bytes, gdn_rc_ckpt_bytes,
    gdn_rc_fwd_workspace_bytes, new_rc_ckpt,
    gdn_strerror, gdn_timing_enable, gdn_timing_read, gdn_version,
    header_functions, load_library, make_shape, new_ckpt,
)
