"""GB300 (sm_103a) local MoE forward: route -> dispatch -> SwiGLU experts -> combine.

The compute lives in ``libmoe.so`` (hand-written CUDA kernels behind the C ABI declared in
``include/moe.h``); ``binding`` marshals torch tensors into that ABI and nothing else.
"""
from .binding import (MoeError, moe_combine_backward, moe_dispatch_backward,  # noqa: F401
                      moe_experts_backward, dispatch_workspace_bytes, experts_workspace_bytes,  # noqa: F401
                      forward_workspace_bytes, moe_combine, moe_device_status, moe_dispatch,
                      moe_experts_forward_dispatched, moe_forward, moe_forward_fused,
                      moe_forward_sigmoid_grouped,
                      moe_forward_with_events, moe_route, moe_route_sigmoid_grouped,
                      moe_selected_router_backward, moe_selected_router_weights,
                      moe_wait_selftest)
