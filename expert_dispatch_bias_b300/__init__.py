"""B300-native (sm_103a) forward pass of a Mixture-of-Experts FFN layer.

The compute lives in ``libmoe.so`` (C ABI: ``include/moe.h``); this package is
its ctypes binding plus buffer helpers.  PyTorch supplies device memory and
streams only.
"""
from ._lib import (  # noqa: F401
    EXPORTS, LAYER_STAGES, LIB_PATH, MOE_BF16, MOE_F32, MOE_OP_BLOCK, MOE_OP_BLOCK_HOST, MOE_OP_FFN, MOE_OP_FFN_FP8,
    MOE_OP_LAYER, MOE_OP_LAYER_FP8, MOE_OP_LOGITS, MOE_OP_FFN_COMBINE, moe_grouped_ffn_fp8, moe_grouped_ffn_gather,
    moe_grouped_ffn_combine, moe_launch_count, moe_layer_forward_fp8, moe_permute_fp8, moe_quantize_fp8,
    MOE_OP_LAYER_HOST, MOE_OP_LAYOUT, MOE_OP_SHARED, MOE_SIGMOID, MOE_SOFTMAX, STATUS, MoeConfig, MoeError,
    MoeLayerOut, MoeLayoutStats, config_from, layer_out, lib, make_config, moe_block_forward,
    moe_block_forward_host, moe_check, moe_combine, moe_combine_add, moe_dispatch_layout, moe_eplb_map,
    moe_eplb_plan, moe_grouped_ffn_mapped, moe_layer_forward_eplb,
    moe_dispatch_layout_static, moe_grouped_ffn, moe_layer_forward, moe_layer_forward_host, moe_permute,
    moe_route, moe_router_logits, moe_rows, moe_shared_ffn, moe_validate_config, moe_workspace_init,
    moe_workspace_size,
)
from .buffers import LayoutBuffers, alloc_layout, alloc_workspace, stats_dict, torch_dtype  # noqa: F401
