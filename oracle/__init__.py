"""CPU oracle for the weight-only-quantized fused MoE layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this package: only the test suite, the package smoke check and the benchmark's
CPU-baseline / reference leg use it.  It shares no code with the CUDA library.

Every function is pinned by checks in the CPU test suite that do not reuse its
own formulas (round trips, closed forms, invariants, brute force on tiny
inputs and hand-worked examples); see the module docstrings for the pins.
"""
from .moe import (  # noqa: F401
    decompress_24,
    dequant_int4,
    dequant_int8,
    dequant_int8_group,
    dequant_layer_expert,
    dequant_linear,
    linear_forward,
    silu,
    expert_ffn,
    moe_forward,
    moe_forward_batches,
    moe_forward_rows,
    moe_align,
    route_topk,
)
