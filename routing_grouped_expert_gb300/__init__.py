"""GB300-native MoE expert-layer forward: route -> permute -> grouped SwiGLU
FFN -> combine, as hand-written sm_103a kernels behind a C ABI (libmoe.so).

The Python layer only marshals arguments: every step runs in the library's
kernels.  Importing the package does not load the library; the first call
does, and raises if libmoe.so has not been built (there is no fallback).
"""
from .binding import (  # noqa: F401
    ForwardGraph,
    MoeError,
    load_library,
    moe_combine,
    moe_diag_wait_timeout,
    moe_diag_count_wait_timeout,
    moe_forward,
    moe_forward_events,
    moe_forward_f32,
    moe_cast_bf16,
    moe_forward_routing,
    moe_forward_stage_name,
    FORWARD_STAGES,
    moe_forward_host,
    moe_forward_train,
    moe_backward,
    moe_workspace_size_train,
    moe_forward_gated,
    moe_router_logits,
    moe_workspace_size_gated,
    moe_get_device_status,
    moe_grouped_ffn,
    moe_permute,
    moe_plan_replicas,
    moe_plan_workspace_size,
    moe_route_topk,
    moe_status_string,
    moe_workspace_size,
    Workspace,
)
