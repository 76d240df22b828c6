"""Seeded synthetic inputs for the weight-quantized fused MoE layer.

This package only *makes inputs*: activations, router outputs (top-k ids and
weights) and quantized expert weights in the library's packed layout. It holds
none of the layer's arithmetic (no dequantization, no GEMM, no activation, no
combine), so both the CUDA library and the CPU oracle can consume what it makes
without sharing any of the method's code. The router outputs come from torch
library calls (softmax / sigmoid, topk); the library's own routing kernel is
checked against the oracle's restatement, not against these.
"""
from .workloads import (  # noqa: F401
    WORKLOADS,
    Workload,
    LayerInputs,
    make_expert_weights,
    make_layer_inputs,
    make_routing,
    make_router_logits,
    routing_params,
    make_hidden,
    make_biases,
    quantize_expert,
    quantize_expert_act_order,
    make_g_idx,
    pack_along_last,
)
