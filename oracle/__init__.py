"""Plain float64 CPU oracle of the weight-quantized fused MoE layer.

TEST INFRASTRUCTURE ONLY. This package is the slow, obviously-correct statement
of what the GPU library computes. Only the test suite, the smoke check and the
CPU-baseline leg of the benchmark import it; the library never does, and this
package imports nothing from the library.
"""
from .wna16_oracle import (  # noqa: F401
    unpack_codes,
    unpack_zeros,
    halfbits_to_f64,
    round_to_halfbits,
    dequantize_expert,
    act_order_permutation,
    AWQ_PACK_ORDER,
    unpack_gptq_qweight,
    unpack_gptq_qzeros,
    unpack_awq,
    align_capacity,
    moe_align_block_size,
    routing_scores,
    routing_group_scores,
    topk_routing,
    silu,
    gated_activation,
    fused_moe_per_token,
    fused_moe_grouped,
)
