"""Single-GPU MoE expert-layer forward for GB300 (sm_103a).

The library is a C ABI (include/moe.h, libmoe_gb300.so built from csrc/);
this package binds it with ctypes.  The shared library is loaded on first
use (or by `load()`); if it has not been built, that raises ImportError --
there is no fallback implementation.
"""
from ._lib import load  # noqa: F401

from .api import (  # noqa: E402,F401
    HostPipeline, LayerDesc, MoEError, MoELayer, desc_for, make_desc, moe_check_status, moe_combine,
    moe_dispatch_layout, moe_expert_gemm1_swiglu, moe_expert_gemm1_swiglu_gather,
    moe_backward, moe_backward_workspace_size, moe_expert_gemm2, moe_expert_gemm2_weighted, moe_combine_slots, moe_forward_host, moe_forward_microbatches, moe_host_workspace_size,
    moe_grouped_swiglu, moe_layout_workspace_size, moe_permute, moe_permute_scatter, moe_route_topk,
    moe_workspace_size, moe_workspace_slot, workspace_view, kernels_per_forward,
    moe_prepare_weights, moe_set_pipeline_wait_limit, moe_set_gemm_pairs, moe_prepare_router,
    moe_set_gemm_tails,
)
