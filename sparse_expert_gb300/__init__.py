"""Single-GPU Mixture-of-Experts layer, forward and backward, for GB300 (sm_103a).

The compute lives in libmoe_gb300.so (hand-written CUDA kernels behind a C
ABI, declared in include/moe_gb300.h); this package is its Python binding.
Importing it fails if the library has not been built.
"""
from ._lib import (  # noqa: F401
    MoEError,
    abi_version,
    forward_intermediates,
    moe_combine,
    moe_combine_backward,
    moe_route_backward,
    moe_dispatch_scan,
    moe_dispatch_scan_noalloc,
    moe_dispatch_workspace_bytes,
    moe_forward,
    moe_forward_host,
    moe_forward_host_stream,
    moe_forward_layout,
    moe_forward_timed,
    moe_forward_routed,
    moe_forward_gathered,
    moe_forward_gathered_timed,
    moe_pack_router_weights,
    moe_router_topk,
    FORWARD_STAGES,
    moe_forward_workspace_bytes,
    moe_grouped_swiglu,
    moe_grouped_gate_up_save,
    moe_grouped_swiglu_backward,
    gu_split,
    moe_backward,
    moe_backward_workspace_bytes,
    moe_backward_timed,
    BACKWARD_STAGES,
    moe_quantize_fp8_blockwise,
    moe_dequantize_fp8_blockwise,
    moe_pack_weights,
    moe_packed_weight_bytes,
    moe_permute,
    moe_read_device_status,
    moe_route_topk,
)
