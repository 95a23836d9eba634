"""Seeded synthetic inputs for the weight-only-quantized MoE layer.

This package is shared by the tests, the oracle's checks and the benchmark.
It draws random weights, activations and router logits, rounds them to the
storage precisions the layer consumes, and runs the offline round-to-nearest
quantizer that turns float weights into the int4/int8 codes and scales the
layer receives.  It holds no part of the layer's own arithmetic (dequantize,
the expert FFN, routing-weighted reduction, token grouping): those live in the
oracle and in the CUDA library, which never import each other.
"""
from .gen import (  # noqa: F401
    WORKLOADS,
    Workload,
    QuantLayer,
    QuantLinear,
    Inputs,
    make_linear,
    make_linear_inputs,
    quantize_int8_24,
    make_layer,
    make_inputs,
    prune_24,
    quantize_int4_24,
    quantize_int4_rtn,
    quantize_int4_rtn_zp,
    quantize_int8_group,
    quantize_int8_rtn,
    round_to,
    round_to_bf16,
    route_topk,
    round_to_f16,
    to_u16_bits,
)
