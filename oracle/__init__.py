"""fp64 CPU oracle for the MoE layer, forward and backward (test infrastructure only).

This package is the checker, not the product.  Only the tests, the smoke
check of ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` use it.
It shares no code with the CUDA path and imports nothing from it.
"""
from .moe_oracle import (  # noqa: F401
    route_topk,
    route_topk_grouped,
    router_topk,
    softmax_rows,
    dispatch,
    permute,
    silu,
    silu_grad,
    expert_mlp,
    expert_mlp_backward,
    expert_gate_up,
    combine,
    combine_backward,
    route_backward,
    moe_forward,
    moe_forward_tokens,
    moe_backward,
)
