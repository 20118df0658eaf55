"""Multi-scale deformable attention core (2D bilinear / 3D trilinear) for NVIDIA B300.

The compute path is libmsda.so (hand-written sm_103a CUDA kernels behind the C ABI in
``include/msda.h``); this package is its thin Python binding, with the same names:

    msda2d_forward, msda2d_backward, msda3d_forward, msda3d_backward,
    msda_query_order, msda2d_forward_ordered, msda3d_forward_ordered,
    msda2d_backward_ordered, msda3d_backward_ordered, msda2d_forward_pruned, msda3d_forward_pruned, msda2d_forward_fused, msda3d_forward_fused,
    msda2d_backward_fused, msda3d_backward_fused, msda_last_error, msda_abi_version,
    msda_build_flags, msda_debug_bounds_status, msda_debug_bounds_selftest

plus ``MSDeformAttnFunction`` / ``ms_deform_attn`` and ``ms_deform_attn_fused``
(torch.autograd) for use inside a model.  The library is
built in-tree by ``python -m scale_deformable_attention_msda3d_b300.build`` (or on first
use when missing); without it every call raises -- there is no CPU fallback.  The same
build writes ``libmsda_debug.so``, which checks every corner row index before its access
(select it with the environment variable MSDA_LIBRARY).
"""
from ._binding import (EXPORTS, MSDA_BF16, MSDA_ERR_CUDA, MSDA_ERR_INTERNAL,  # noqa: F401
                       MSDA_ERR_INVALID_ARG, MSDA_ERR_UNSUPPORTED, MSDA_F32, MSDA_MAX_LEVELS,
                       MSDA_MAX_POINTS, MSDA_OK, MSDA_BUILD_DEBUG_BOUNDS, MsdaError,
                       backward_raw, backward_ordered_raw, forward_ordered_raw,
                       msda2d_backward_ordered, msda3d_backward_ordered, msda_build_flags,
                       msda_debug_bounds_status, msda_debug_bounds_selftest,
                       forward_pruned_raw, msda2d_forward_pruned, msda3d_forward_pruned,
                       forward_fused_raw, msda2d_forward_fused, msda3d_forward_fused,
                       backward_fused_raw, msda2d_backward_fused, msda3d_backward_fused,
                       forward_raw, library_path, load, make_dims, msda2d_backward,
                       msda2d_forward, msda2d_forward_ordered, msda3d_backward,
                       msda3d_forward, msda3d_forward_ordered, msda_abi_version, msda_dims,
                       msda_last_error, msda_query_order, query_order_raw, query_order_static_raw,
                       query_order_workspace_bytes, query_order_workspace_raw)
from .autograd import MSDeformAttnFunction, ms_deform_attn, ms_deform_attn_fused  # noqa: F401
