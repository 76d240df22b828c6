"""Fused weight-only-quantized (W4A16 / W8A16) Mixture-of-Experts layer for one
GB300 GPU: a C-ABI CUDA library (``include/wna16_moe.h``) and its binding.
"""
from .binding import (  # noqa: F401
    DEV_BAD_EXPERT_ID,
    DEV_BAD_GROUPS,
    DEV_TIMEOUT,
    EXPORTED,
    PackedWeights,
    Plan,
    act_order_prepare,
    WNA16Error,
    align_capacity,
    check_launch_plan,
    check_wait_timeout,
    choose_block,
    convert_checkpoint,
    fused_moe,
    fused_moe_noalloc,
    fused_moe_prepacked,
    fused_moe_routed,
    load,
    moe_align_block_size,
    noalloc_read_status,
    prepack,
    read_device_status,
    topk_routing,
    workspace_bytes,
)
from .build import LIB, build  # noqa: F401
