"""ctypes binding of libqmoe (include/qmoe.h): argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; PyTorch supplies
device memory and the current stream.  There is no fallback: if the library
is not built, or a call fails, an exception says so.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_int64, c_size_t, c_uint8, c_uint16, c_void_p

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libqmoe.so")
HEADER_PATH = os.path.join(os.path.dirname(HERE), "include", "qmoe.h")

QMOE_OK = 0
QMOE_ERR_INVALID_ARG = 1
QMOE_ERR_UNSUPPORTED = 2
QMOE_ERR_DEVICE_MISMATCH = 3
QMOE_ERR_WORKSPACE = 4
QMOE_ERR_CUDA = 5
QMOE_ERR_TIMEOUT = 6
QMOE_ERR_BAD_EXPERT_ID = 7

QMOE_INT4_GROUP = 1
QMOE_INT8_PER_COL = 2
QMOE_INT4_GROUP_ZP = 3
QMOE_INT8_GROUP = 4
QMOE_INT4_GROUP_24 = 5
QMOE_INT8_24 = 6
QMOE_F16 = 1
QMOE_BF16 = 2
QMOE_F32 = 3


class QmoeLayer(ctypes.Structure):
    _fields_ = [
        ("E", c_int32), ("H", c_int32), ("I", c_int32), ("group_size", c_int32),
        ("qt", c_int32), ("act_dtype", c_int32), ("scale_dtype", c_int32),
        ("w13", c_void_p), ("w2", c_void_p), ("s13", c_void_p), ("s2", c_void_p), ("perm13", c_void_p),
    ]


class QmoeLinear(ctypes.Structure):
    _fields_ = [
        ("N", c_int32), ("K", c_int32), ("group_size", c_int32), ("qt", c_int32), ("act_dtype", c_int32),
        ("scale_dtype", c_int32), ("w", c_void_p), ("s", c_void_p), ("perm", c_void_p),
    ]


class QmoePlanInfo(ctypes.Structure):
    _fields_ = [("token_tile", c_int32), ("issuers", c_int32), ("acc_bufs", c_int32), ("split1", c_int32),
                ("split2", c_int32), ("w_stages", c_int32), ("ab_stages", c_int32), ("stage_bytes", c_int32),
                ("workspace_bytes", c_int64), ("b_stages", c_int32), ("dq_sets", c_int32),
                ("cta_pair", c_int32), ("cta_pair_down", c_int32), ("reserved", c_int32 * 2)]


class QmoeOptions(ctypes.Structure):
    _fields_ = [("split1", c_int32), ("split2", c_int32), ("token_tile", c_int32), ("fault_injection", c_int32),
                ("issuers", c_int32), ("token_ring", c_int32), ("dq_sets", c_int32),
                ("weight_l2", c_int32), ("int4_group_epilogue", c_int32), ("topk_reduce", c_int32),
                ("cta_pair", c_int32), ("reserved", c_int32 * 5)]


class QmoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib = None

_SIGS = {
    "qmoe_abi_version": (c_int32, []),
    "qmoe_status_string": (ctypes.c_char_p, [c_int32]),
    "qmoe_packed_bytes": (c_size_t, [c_int32, c_int32, c_int32, c_int32, c_int32]),
    "qmoe_pack_int4": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_int32,
                                 POINTER(c_uint8), POINTER(c_uint16), POINTER(c_int32),
                                 POINTER(c_uint8), POINTER(c_uint16), POINTER(c_int32),
                                 c_void_p, c_void_p, POINTER(c_int32)]),
    "qmoe_unpack_int4": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p,
                                   POINTER(c_int32), POINTER(c_int32),
                                   POINTER(c_uint8), POINTER(c_uint16), POINTER(c_uint8), POINTER(c_uint16)]),
    "qmoe_pack_int4_zp": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_int32,
                                    POINTER(c_uint8), POINTER(c_uint16), POINTER(c_uint8), POINTER(c_int32),
                                    POINTER(c_uint8), POINTER(c_uint16), POINTER(c_uint8), POINTER(c_int32),
                                    c_void_p, c_void_p, POINTER(c_int32)]),
    "qmoe_unpack_int4_zp": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p,
                                      POINTER(c_int32), POINTER(c_int32),
                                      POINTER(c_uint8), POINTER(c_uint16), POINTER(c_uint8),
                                      POINTER(c_uint8), POINTER(c_uint16), POINTER(c_uint8)]),
    "qmoe_pack_int8_group": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_void_p, POINTER(c_uint16), c_void_p,
                                       POINTER(c_uint16), c_void_p, c_void_p]),
    "qmoe_pack_int4_24": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_int32, POINTER(c_uint8), POINTER(c_uint16),
                                    POINTER(c_uint8), POINTER(c_uint16), c_void_p, c_void_p]),
    "qmoe_unpack_int4_24": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p, POINTER(c_uint8),
                                      POINTER(c_uint16), POINTER(c_uint8), POINTER(c_uint16)]),
    "qmoe_unpack_int8_group": (c_int32, [c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p, POINTER(c_uint16),
                                         c_void_p, POINTER(c_uint16)]),
    "qmoe_pack_int8": (c_int32, [c_int32, c_int32, c_int32, c_void_p, POINTER(c_float), c_void_p, POINTER(c_float),
                                 c_void_p, POINTER(c_float), c_void_p, POINTER(c_float)]),
    "qmoe_unpack_int8": (c_int32, [c_int32, c_int32, c_int32, c_void_p, POINTER(c_float), c_void_p, POINTER(c_float),
                                   c_void_p, POINTER(c_float), c_void_p, POINTER(c_float)]),
    "qmoe_moe_align": (c_int32, [c_void_p, c_int64, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                 c_int64, c_void_p]),
    "qmoe_workspace_size": (c_size_t, [POINTER(QmoeLayer), c_int64, c_int32]),
    "qmoe_workspace_size_ex": (c_size_t, [POINTER(QmoeLayer), c_int64, c_int32, POINTER(QmoeOptions)]),
    "qmoe_describe_plan": (c_int32, [POINTER(QmoeLayer), c_int64, c_int32, POINTER(QmoeOptions), c_int32,
                                     POINTER(QmoePlanInfo)]),
    "qmoe_forward": (c_int32, [POINTER(QmoeLayer), c_void_p, c_int64, c_void_p, c_void_p, c_int32, c_void_p,
                               c_void_p, c_size_t, c_void_p]),
    "qmoe_forward_ex": (c_int32, [POINTER(QmoeLayer), c_void_p, c_int64, c_void_p, c_void_p, c_int32, c_void_p,
                                  c_void_p, c_size_t, c_void_p, POINTER(QmoeOptions)]),
    "qmoe_forward_profiled": (c_int32, [POINTER(QmoeLayer), c_void_p, c_int64, c_void_p, c_void_p, c_int32,
                                        c_void_p, c_void_p, c_size_t, c_void_p, POINTER(QmoeOptions),
                                        POINTER(c_void_p), c_int32, POINTER(c_int32)]),
    "qmoe_workspace_size_host": (c_size_t, [POINTER(QmoeLayer), c_int64, c_int32]),
    "qmoe_forward_host": (c_int32, [POINTER(QmoeLayer), c_void_p, c_int64, c_void_p, c_void_p, c_int32, c_void_p,
                                    c_void_p, c_size_t, c_void_p]),
    "qmoe_read_device_status": (c_int32, [c_void_p, c_void_p]),
    "qmoe_route_topk": (c_int32, [c_void_p, c_int32, c_int64, c_int32, c_int32, c_int32, c_void_p, c_void_p,
                                  c_void_p]),
    "qmoe_workspace_size_logits": (c_size_t, [POINTER(QmoeLayer), c_int64, c_int32]),
    "qmoe_forward_logits": (c_int32, [POINTER(QmoeLayer), c_void_p, c_int64, c_void_p, c_int32, c_int32, c_int32,
                                      c_void_p, c_void_p, c_size_t, c_void_p]),
    "qmoe_forward_noalloc": (c_int32, [POINTER(QmoeLayer), c_void_p, c_int64, c_void_p, c_void_p, c_int32,
                                       c_void_p, c_void_p]),
    "qmoe_read_noalloc_status": (c_int32, [c_void_p]),
    "qmoe_pack_int8_24": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_void_p, POINTER(c_float), c_void_p, POINTER(c_float)]),
    "qmoe_unpack_int8_24": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_void_p, POINTER(c_float), c_void_p,
                                      POINTER(c_float), c_void_p, c_void_p, c_void_p, c_void_p]),
    "qmoe_pack_linear": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                   c_void_p, c_void_p, POINTER(c_float), c_void_p]),
    "qmoe_unpack_linear": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_void_p, POINTER(c_float), c_void_p,
                                     c_void_p, c_void_p, c_void_p]),
    "qmoe_linear_workspace_size": (c_size_t, [POINTER(QmoeLinear), c_int64, POINTER(QmoeOptions)]),
    "qmoe_linear_describe_plan": (c_int32, [POINTER(QmoeLinear), c_int64, POINTER(QmoeOptions), c_int32,
                                            POINTER(QmoePlanInfo)]),
    "qmoe_linear_forward": (c_int32, [POINTER(QmoeLinear), c_void_p, c_int64, c_void_p, c_void_p, c_size_t, c_void_p,
                                      POINTER(QmoeOptions)]),
}


def lib():
    """The loaded libqmoe (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libqmoe is not built ({LIB_PATH} missing); build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` or weight_only_quantized_moe_gb300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().qmoe_status_string(int(status)).decode()


def check(status: int, where: str):
    if status != QMOE_OK:
        raise QmoeError(status, where)
