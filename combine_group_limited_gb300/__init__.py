"""MoE expert-parallel dispatch/combine on one GB300 (sm_103a).

The hot path -- group-limited top-k gating, dispatch layout, BF16/FP8
permute-scatter, inverse gather and weighted combine -- runs in the CUDA
kernels of ``libep_gb300.so`` behind the C ABI of ``include/ep.h``.  This
package is its thin Python binding (names follow the C entry points) plus the
in-tree build step.
"""
from ._binding import (  # noqa: F401
    EP_DTYPE_BF16, EP_DTYPE_FP8_E4M3_B128, EP_ERR_ALIGNMENT, EP_ERR_CUDA, EP_ERR_INVALID_ARG, EP_ERR_UNSUPPORTED,
    EP_DTYPE_MXFP8_E4M3_B32, EP_FLAG_BAD_EXPERT, EP_FLAG_BAD_ROW, EP_FLAG_TIMEOUT, EP_OK, EP_SCORE_RAW, EP_SCORE_SOFTMAX, EXPORTS,
    CapLayout, EpError, GateCfg, Layout, alloc_layout, alloc_layout_workspace, ep_combine, ep_combine_backward,
    ep_combine_fp8, ep_decode_dispatch, ep_dispatch, ep_dispatch_backward, ep_gate, ep_get_layout, ep_get_layout_capacity,
    ep_gate_layout, ep_get_layout_noalloc, ep_layout_workspace_bytes, ep_selftest_grid_barrier, gate_cfg, load,
    status_str)
