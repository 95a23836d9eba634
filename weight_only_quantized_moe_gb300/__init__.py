"""GB300-native fused mixture-of-experts layer with weight-only-quantized experts.

W4A16 (GPTQ-style int4, group 128, optional act-order) and W8A16 (per-column
int8) expert weights are dequantized on the fly inside hand-written sm_103a
tcgen05 GEMMs; the C ABI is include/qmoe.h, the kernels live in csrc/.
"""
from ._native import (  # noqa: F401
    HEADER_PATH,
    LIB_PATH,
    QMOE_ERR_BAD_EXPERT_ID,
    QMOE_ERR_CUDA,
    QMOE_ERR_DEVICE_MISMATCH,
    QMOE_ERR_INVALID_ARG,
    QMOE_ERR_TIMEOUT,
    QMOE_ERR_UNSUPPORTED,
    QMOE_ERR_WORKSPACE,
    QMOE_OK,
    QmoeError,
    lib,
    status_string,
)
from .api import (  # noqa: F401
    DeviceLayer,
    alloc_workspace,
    default_group_size,
    make_options,
    packed_bytes,
    qmoe_forward,
    qmoe_forward_host,
    qmoe_forward_logits,
    qmoe_forward_noalloc,
    qmoe_read_noalloc_status,
    qmoe_forward_profiled,
    qmoe_moe_align,
    qmoe_pack_int4,
    qmoe_pack_int8,
    qmoe_pack_int8_group,
    qmoe_pack_int4_24,
    qmoe_read_device_status,
    qmoe_route_topk,
    qmoe_unpack_int4,
    qmoe_unpack_int8_group,
    qmoe_unpack_int4_24,
    qmoe_workspace_size_logits,
    qmoe_unpack_int8,
    qmoe_workspace_size,
    qmoe_describe_plan,
    qmoe_workspace_size_host,
)
