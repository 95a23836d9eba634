"""Python face of libqmoe with the C ABI's names (argument marshalling only).

Host packing takes and returns numpy arrays; the forward and moe_align take
torch CUDA tensors and run on the current torch stream unless one is given.
"""
from __future__ import annotations

from ctypes import POINTER, byref, c_float, c_int32, c_uint8, c_uint16, c_void_p

import numpy as np
import torch

from . import _native as N

_ACT = {"f16": N.QMOE_F16, "bf16": N.QMOE_BF16}
_TORCH_ACT = {"f16": torch.float16, "bf16": torch.bfloat16}
_QT = {"int4": N.QMOE_INT4_GROUP, "int4zp": N.QMOE_INT4_GROUP_ZP, "int8": N.QMOE_INT8_PER_COL,
       "int8g": N.QMOE_INT8_GROUP, "int4s24": N.QMOE_INT4_GROUP_24, "int8s24": N.QMOE_INT8_24}


def default_group_size(qt: str) -> int:
    return -1 if qt in ("int8", "int8s24") else 128


def _np_ptr(a, ctype):
    return None if a is None else a.ctypes.data_as(POINTER(ctype))


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream)


def packed_bytes(qt: str, E: int, rows: int, K: int, group_size: int | None = None) -> int:
    gs = default_group_size(qt) if group_size is None else group_size
    return int(N.lib().qmoe_packed_bytes(_QT[qt], E, rows, K, gs))


# ----------------------------------------------------------------------------
# packing (host)
# ----------------------------------------------------------------------------
def qmoe_pack_int4(E, H, I, scale_dtype, q13, s13_bits, g13, q2, s2_bits, g2, group_size=128, z13=None, z2=None):
    """Pack canonical int4 weights (see include/qmoe.h).  Scales are uint16 bit
    patterns [E, K/G, N] ([E, 1, N] with group_size -1); zero points z13/z2
    (uint8, same shapes) select the asymmetric format (qmoe_pack_int4_zp)."""
    q13 = np.ascontiguousarray(q13, np.uint8)
    q2 = np.ascontiguousarray(q2, np.uint8)
    s13_bits = np.ascontiguousarray(s13_bits, np.uint16)
    s2_bits = np.ascontiguousarray(s2_bits, np.uint16)
    g13 = None if g13 is None else np.ascontiguousarray(g13, np.int32)
    g2 = None if g2 is None else np.ascontiguousarray(g2, np.int32)
    qt = "int4" if z13 is None else "int4zp"
    w13 = np.empty(packed_bytes(qt, E, 2 * I, H, group_size), np.uint8)
    w2 = np.empty(packed_bytes(qt, E, H, I, group_size), np.uint8)
    perm13 = np.empty((E, H), np.int32) if g13 is not None else None
    if z13 is None:
        st = N.lib().qmoe_pack_int4(E, H, I, group_size, _ACT[scale_dtype], _np_ptr(q13, c_uint8),
                                    _np_ptr(s13_bits, c_uint16), _np_ptr(g13, c_int32), _np_ptr(q2, c_uint8),
                                    _np_ptr(s2_bits, c_uint16), _np_ptr(g2, c_int32), w13.ctypes.data_as(c_void_p),
                                    w2.ctypes.data_as(c_void_p), _np_ptr(perm13, c_int32))
        N.check(st, "qmoe_pack_int4")
    else:
        z13 = np.ascontiguousarray(z13, np.uint8)
        z2 = np.ascontiguousarray(z2, np.uint8)
        st = N.lib().qmoe_pack_int4_zp(E, H, I, group_size, _ACT[scale_dtype], _np_ptr(q13, c_uint8),
                                       _np_ptr(s13_bits, c_uint16), _np_ptr(z13, c_uint8), _np_ptr(g13, c_int32),
                                       _np_ptr(q2, c_uint8), _np_ptr(s2_bits, c_uint16), _np_ptr(z2, c_uint8),
                                       _np_ptr(g2, c_int32), w13.ctypes.data_as(c_void_p),
                                       w2.ctypes.data_as(c_void_p), _np_ptr(perm13, c_int32))
        N.check(st, "qmoe_pack_int4_zp")
    return {"w13": w13, "w2": w2, "perm13": perm13}


def qmoe_unpack_int4(E, H, I, w13, w2, g13, g2, group_size=128, zp=False):
    """Inverse of qmoe_pack_int4: (q13, s13, q2, s2), plus (z13, z2) when ``zp``."""
    n13 = 1 if group_size < 0 else H // 128
    n2 = 1 if group_size < 0 else I // 128
    q13 = np.empty((E, 2 * I, H), np.uint8)
    s13 = np.empty((E, n13, 2 * I), np.uint16)
    q2 = np.empty((E, H, I), np.uint8)
    s2 = np.empty((E, n2, H), np.uint16)
    g13 = None if g13 is None else np.ascontiguousarray(g13, np.int32)
    g2 = None if g2 is None else np.ascontiguousarray(g2, np.int32)
    if not zp:
        st = N.lib().qmoe_unpack_int4(E, H, I, group_size, w13.ctypes.data_as(c_void_p), w2.ctypes.data_as(c_void_p),
                                      _np_ptr(g13, c_int32), _np_ptr(g2, c_int32), _np_ptr(q13, c_uint8),
                                      _np_ptr(s13, c_uint16), _np_ptr(q2, c_uint8), _np_ptr(s2, c_uint16))
        N.check(st, "qmoe_unpack_int4")
        return q13, s13, q2, s2
    z13 = np.empty((E, n13, 2 * I), np.uint8)
    z2 = np.empty((E, n2, H), np.uint8)
    st = N.lib().qmoe_unpack_int4_zp(E, H, I, group_size, w13.ctypes.data_as(c_void_p), w2.ctypes.data_as(c_void_p),
                                     _np_ptr(g13, c_int32), _np_ptr(g2, c_int32), _np_ptr(q13, c_uint8),
                                     _np_ptr(s13, c_uint16), _np_ptr(z13, c_uint8), _np_ptr(q2, c_uint8),
                                     _np_ptr(s2, c_uint16), _np_ptr(z2, c_uint8))
    N.check(st, "qmoe_unpack_int4_zp")
    return q13, s13, q2, s2, z13, z2


def qmoe_pack_int8_group(E, H, I, scale_dtype, q13, s13_bits, q2, s2_bits):
    """Pack canonical group-128 int8 weights (scales as uint16 bit patterns [E, K/128, N])."""
    q13 = np.ascontiguousarray(q13, np.int8)
    q2 = np.ascontiguousarray(q2, np.int8)
    s13_bits = np.ascontiguousarray(s13_bits, np.uint16)
    s2_bits = np.ascontiguousarray(s2_bits, np.uint16)
    w13 = np.empty(packed_bytes("int8g", E, 2 * I, H), np.uint8)
    w2 = np.empty(packed_bytes("int8g", E, H, I), np.uint8)
    st = N.lib().qmoe_pack_int8_group(E, H, I, _ACT[scale_dtype], q13.ctypes.data_as(c_void_p),
                                      _np_ptr(s13_bits, c_uint16), q2.ctypes.data_as(c_void_p),
                                      _np_ptr(s2_bits, c_uint16), w13.ctypes.data_as(c_void_p),
                                      w2.ctypes.data_as(c_void_p))
    N.check(st, "qmoe_pack_int8_group")
    return {"w13": w13, "w2": w2}


def qmoe_unpack_int8_group(E, H, I, w13, w2):
    q13 = np.empty((E, 2 * I, H), np.int8)
    s13 = np.empty((E, H // 128, 2 * I), np.uint16)
    q2 = np.empty((E, H, I), np.int8)
    s2 = np.empty((E, I // 128, H), np.uint16)
    st = N.lib().qmoe_unpack_int8_group(E, H, I, w13.ctypes.data_as(c_void_p), w2.ctypes.data_as(c_void_p),
                                        q13.ctypes.data_as(c_void_p), _np_ptr(s13, c_uint16),
                                        q2.ctypes.data_as(c_void_p), _np_ptr(s2, c_uint16))
    N.check(st, "qmoe_unpack_int8_group")
    return q13, s13, q2, s2


def qmoe_pack_int4_24(E, H, I, scale_dtype, q13, s13_bits, q2, s2_bits, group_size=128):
    """Pack 2:4-sparse int4: dense codes (8 at the pruned channels, at most 2
    other codes per aligned group of 4 input channels) and uint16 scale bit
    patterns [E, K/G, N] ([E, 1, N] with group_size -1)."""
    q13 = np.ascontiguousarray(q13, np.uint8)
    q2 = np.ascontiguousarray(q2, np.uint8)
    s13_bits = np.ascontiguousarray(s13_bits, np.uint16)
    s2_bits = np.ascontiguousarray(s2_bits, np.uint16)
    w13 = np.empty(packed_bytes("int4s24", E, 2 * I, H, group_size), np.uint8)
    w2 = np.empty(packed_bytes("int4s24", E, H, I, group_size), np.uint8)
    st = N.lib().qmoe_pack_int4_24(E, H, I, group_size, _ACT[scale_dtype], _np_ptr(q13, c_uint8),
                                   _np_ptr(s13_bits, c_uint16), _np_ptr(q2, c_uint8), _np_ptr(s2_bits, c_uint16),
                                   w13.ctypes.data_as(c_void_p), w2.ctypes.data_as(c_void_p))
    N.check(st, "qmoe_pack_int4_24")
    return {"w13": w13, "w2": w2}


def qmoe_unpack_int4_24(E, H, I, w13, w2, group_size=128):
    """Inverse of qmoe_pack_int4_24: dense (q13, s13, q2, s2)."""
    n13 = 1 if group_size < 0 else H // 128
    n2 = 1 if group_size < 0 else I // 128
    q13 = np.empty((E, 2 * I, H), np.uint8)
    s13 = np.empty((E, n13, 2 * I), np.uint16)
    q2 = np.empty((E, H, I), np.uint8)
    s2 = np.empty((E, n2, H), np.uint16)
    st = N.lib().qmoe_unpack_int4_24(E, H, I, group_size, w13.ctypes.data_as(c_void_p), w2.ctypes.data_as(c_void_p),
                                     _np_ptr(q13, c_uint8), _np_ptr(s13, c_uint16), _np_ptr(q2, c_uint8),
                                     _np_ptr(s2, c_uint16))
    N.check(st, "qmoe_unpack_int4_24")
    return q13, s13, q2, s2


def _float_scales(qt: str, group_size: int) -> bool:
    """Formats whose scales are float32, one per output feature (applied to the accumulator)."""
    return qt == "int8" or (qt == "int8s24" and group_size == -1)


def qmoe_pack_int8_24(E, H, I, scale_dtype, q13, s13, q2, s2, group_size=-1):
    """Pack 2:4-sparse int8: dense codes (0 at the pruned channels).  group_size -1:
    float32 scales [E, N] (scale_dtype "f32"); 128: uint16 bit patterns [E, K/128, N]."""
    q13 = np.ascontiguousarray(q13, np.int8)
    q2 = np.ascontiguousarray(q2, np.int8)
    cw = group_size == -1
    sdt = np.float32 if cw else np.uint16
    s13 = np.ascontiguousarray(s13, sdt)
    s2 = np.ascontiguousarray(s2, sdt)
    w13 = np.empty(packed_bytes("int8s24", E, 2 * I, H, group_size), np.uint8)
    w2 = np.empty(packed_bytes("int8s24", E, H, I, group_size), np.uint8)
    s13p = np.empty((E, 2 * I), np.float32) if cw else None
    s2p = np.empty((E, H), np.float32) if cw else None
    st = N.lib().qmoe_pack_int8_24(E, H, I, group_size, N.QMOE_F32 if cw else _ACT[scale_dtype],
                                   q13.ctypes.data_as(c_void_p), s13.ctypes.data_as(c_void_p),
                                   q2.ctypes.data_as(c_void_p), s2.ctypes.data_as(c_void_p),
                                   w13.ctypes.data_as(c_void_p), _np_ptr(s13p, c_float), w2.ctypes.data_as(c_void_p),
                                   _np_ptr(s2p, c_float))
    N.check(st, "qmoe_pack_int8_24")
    return {"w13": w13, "w2": w2, "s13": s13p, "s2": s2p}


def qmoe_unpack_int8_24(E, H, I, w13, s13p, w2, s2p, group_size=-1):
    """Inverse of qmoe_pack_int8_24: dense (q13, s13, q2, s2)."""
    cw = group_size == -1
    q13 = np.empty((E, 2 * I, H), np.int8)
    q2 = np.empty((E, H, I), np.int8)
    s13 = np.empty((E, 2 * I), np.float32) if cw else np.empty((E, H // 128, 2 * I), np.uint16)
    s2 = np.empty((E, H), np.float32) if cw else np.empty((E, I // 128, H), np.uint16)
    st = N.lib().qmoe_unpack_int8_24(E, H, I, group_size, w13.ctypes.data_as(c_void_p), _np_ptr(s13p, c_float),
                                     w2.ctypes.data_as(c_void_p), _np_ptr(s2p, c_float), q13.ctypes.data_as(c_void_p),
                                     s13.ctypes.data_as(c_void_p), q2.ctypes.data_as(c_void_p),
                                     s2.ctypes.data_as(c_void_p))
    N.check(st, "qmoe_unpack_int8_24")
    return q13, s13, q2, s2


def qmoe_pack_linear(qt, N_out, K, act, q, s, group_size=None, z=None, g_idx=None):
    """Pack one [N, K] weight matrix for the dense linear layer (see include/qmoe.h).
    int4 formats: q uint8, s float32 [K/G or 1, N] exact in ``act``; int8 group / 2:4
    group: q int8, s float32 [K/128, N]; per-column formats: q int8, s float32 [N]."""
    gs = default_group_size(qt) if group_size is None else group_size
    fs = _float_scales(qt, gs)
    qa = np.ascontiguousarray(q, np.uint8 if qt.startswith("int4") else np.int8)
    sa = np.ascontiguousarray(s, np.float32) if fs else _scale_bits(s, act)
    za = None if z is None else np.ascontiguousarray(z, np.uint8)
    ga = None if g_idx is None else np.ascontiguousarray(g_idx, np.int32)
    w = np.empty(packed_bytes(qt, 1, N_out, K, gs), np.uint8)
    sp = np.empty(N_out, np.float32) if fs else None
    perm = np.empty(K, np.int32) if ga is not None else None
    st = N.lib().qmoe_pack_linear(_QT[qt], N_out, K, gs, N.QMOE_F32 if fs else _ACT[act], qa.ctypes.data_as(c_void_p),
                                  sa.ctypes.data_as(c_void_p), _np_ptr(za, c_uint8), _np_ptr(ga, c_int32),
                                  w.ctypes.data_as(c_void_p), _np_ptr(sp, c_float), _np_ptr(perm, c_int32))
    N.check(st, "qmoe_pack_linear")
    return {"w": w, "s": sp, "perm": perm}


def qmoe_unpack_linear(qt, N_out, K, packed, group_size=None, g_idx=None):
    """Inverse of qmoe_pack_linear: (q, s) with s as uint16 bits or float32, plus z for int4zp."""
    gs = default_group_size(qt) if group_size is None else group_size
    fs = _float_scales(qt, gs)
    ng = 1 if gs < 0 else K // 128
    q = np.empty((N_out, K), np.uint8 if qt.startswith("int4") else np.int8)
    s = np.empty(N_out, np.float32) if fs else np.empty((ng, N_out), np.uint16)
    z = np.empty((ng, N_out), np.uint8) if qt == "int4zp" else None
    ga = None if g_idx is None else np.ascontiguousarray(g_idx, np.int32)
    st = N.lib().qmoe_unpack_linear(_QT[qt], N_out, K, gs, packed["w"].ctypes.data_as(c_void_p),
                                    _np_ptr(packed.get("s"), c_float), _np_ptr(ga, c_int32), q.ctypes.data_as(c_void_p),
                                    s.ctypes.data_as(c_void_p), _np_ptr(z, c_uint8))
    N.check(st, "qmoe_unpack_linear")
    return (q, s, z) if z is not None else (q, s)


def qmoe_pack_int8(E, H, I, q13, s13, q2, s2):
    q13 = np.ascontiguousarray(q13, np.int8)
    q2 = np.ascontiguousarray(q2, np.int8)
    s13 = np.ascontiguousarray(s13, np.float32)
    s2 = np.ascontiguousarray(s2, np.float32)
    w13 = np.empty(packed_bytes("int8", E, 2 * I, H), np.uint8)
    w2 = np.empty(packed_bytes("int8", E, H, I), np.uint8)
    s13p = np.empty((E, 2 * I), np.float32)
    s2p = np.empty((E, H), np.float32)
    st = N.lib().qmoe_pack_int8(E, H, I, q13.ctypes.data_as(c_void_p), _np_ptr(s13, c_float),
                                q2.ctypes.data_as(c_void_p), _np_ptr(s2, c_float), w13.ctypes.data_as(c_void_p),
                                _np_ptr(s13p, c_float), w2.ctypes.data_as(c_void_p), _np_ptr(s2p, c_float))
    N.check(st, "qmoe_pack_int8")
    return {"w13": w13, "w2": w2, "s13": s13p, "s2": s2p}


def qmoe_unpack_int8(E, H, I, w13, s13p, w2, s2p):
    q13 = np.empty((E, 2 * I, H), np.int8)
    s13 = np.empty((E, 2 * I), np.float32)
    q2 = np.empty((E, H, I), np.int8)
    s2 = np.empty((E, H), np.float32)
    st = N.lib().qmoe_unpack_int8(E, H, I, w13.ctypes.data_as(c_void_p), _np_ptr(s13p, c_float),
                                  w2.ctypes.data_as(c_void_p), _np_ptr(s2p, c_float), q13.ctypes.data_as(c_void_p),
                                  _np_ptr(s13, c_float), q2.ctypes.data_as(c_void_p), _np_ptr(s2, c_float))
    N.check(st, "qmoe_unpack_int8")
    return q13, s13, q2, s2


def _scale_bits(s: np.ndarray, act: str) -> np.ndarray:
    """uint16 bit patterns of float32 scales that are exact in the activation type."""
    t = torch.from_numpy(np.ascontiguousarray(s, np.float32)).to(_TORCH_ACT[act])
    return t.view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------------------
# device layer
# ----------------------------------------------------------------------------
class DeviceLayer:
    """A packed layer resident on one CUDA device plus its C descriptor."""

    def __init__(self, qt, E, H, I, act, w13, w2, s13=None, s2=None, perm13=None, group_size=None):
        self.qt, self.E, self.H, self.I, self.act = qt, E, H, I, act
        self.group_size = default_group_size(qt) if group_size is None else group_size
        self.w13, self.w2, self.s13, self.s2, self.perm13 = w13, w2, s13, s2, perm13
        self.struct = N.QmoeLayer(
            E, H, I, self.group_size, _QT[qt], _ACT[act],
            N.QMOE_F32 if _float_scales(qt, self.group_size) else _ACT[act],
            w13.data_ptr(), w2.data_ptr(),
            None if s13 is None else s13.data_ptr(), None if s2 is None else s2.data_ptr(),
            None if perm13 is None else perm13.data_ptr())

    @property
    def torch_dtype(self):
        return _TORCH_ACT[self.act]

    def weight_bytes(self) -> int:
        n = self.w13.numel() + self.w2.numel()
        if self.s13 is not None:
            n += 4 * (self.s13.numel() + self.s2.numel())
        return n

    @classmethod
    def from_packed(cls, qt, E, H, I, act, packed, device="cuda", group_size=None):
        def dev(a, dt=None):
            if a is None:
                return None
            return torch.from_numpy(np.ascontiguousarray(a)).to(device)
        gs = default_group_size(qt) if group_size is None else group_size
        fs = _float_scales(qt, gs)
        return cls(qt, E, H, I, act, dev(packed["w13"]), dev(packed["w2"]),
                   dev(packed.get("s13")) if fs else None,
                   dev(packed.get("s2")) if fs else None,
                   dev(packed.get("perm13")), gs)

    @classmethod
    def from_canonical(cls, qt, act, q13, s13, q2, s2, g13=None, g2=None, device="cuda", z13=None, z2=None,
                       group_size=None):
        """Pack canonical codes/scales on the host and upload them.

        int4 / int4zp: q uint8 codes, s float32 [E, K/G, N] (exact in ``act``;
        G = K for group_size -1), g int32 or None, int4zp zero points z uint8
        like s.  int4s24: as int4 without g, codes 2:4 sparse along K.  int8: q
        int8 codes, s float32 [E, N].  int8g: q int8 codes, s float32
        [E, K/128, N] (exact in ``act``).
        """
        E, N2, H = q13.shape
        I = N2 // 2
        gs = default_group_size(qt) if group_size is None else group_size
        if qt in ("int4", "int4zp"):
            packed = qmoe_pack_int4(E, H, I, act, q13, _scale_bits(s13, act), g13, q2, _scale_bits(s2, act), g2,
                                    gs, z13 if qt == "int4zp" else None, z2 if qt == "int4zp" else None)
        elif qt == "int4s24":
            packed = qmoe_pack_int4_24(E, H, I, act, q13, _scale_bits(s13, act), q2, _scale_bits(s2, act), gs)
        elif qt == "int8g":
            packed = qmoe_pack_int8_group(E, H, I, act, q13, _scale_bits(s13, act), q2, _scale_bits(s2, act))
        elif qt == "int8s24":
            if gs == -1:
                packed = qmoe_pack_int8_24(E, H, I, "f32", q13, s13, q2, s2, -1)
            else:
                packed = qmoe_pack_int8_24(E, H, I, act, q13, _scale_bits(s13, act), q2, _scale_bits(s2, act), gs)
        else:
            packed = qmoe_pack_int8(E, H, I, q13, s13, q2, s2)
        return cls.from_packed(qt, E, H, I, act, packed, device, gs)


# ----------------------------------------------------------------------------
# device entry points
# ----------------------------------------------------------------------------
def make_options(split1=0, split2=0, token_tile=0, fault_injection=0, issuers=0, token_ring=0, dq_sets=0,
                 weight_l2=0, int4_group_epilogue=0, topk_reduce=0, cta_pair=0):
    return N.QmoeOptions(split1, split2, token_tile, fault_injection, issuers, token_ring, dq_sets, weight_l2,
                         int4_group_epilogue, topk_reduce, cta_pair)


def qmoe_moe_align(topk_ids: torch.Tensor, E: int, block: int, capacity: int | None = None, stream=None):
    assert topk_ids.is_cuda and topk_ids.dtype == torch.int32 and topk_ids.is_contiguous()
    M, k = topk_ids.shape
    P = M * k
    if capacity is None:
        capacity = P + E * (block - 1)
    dev = topk_ids.device
    sorted_ids = torch.empty(max(capacity, 1), dtype=torch.int32, device=dev)
    expert_ids = torch.empty(max(-(-capacity // block), 1), dtype=torch.int32, device=dev)
    npp = torch.empty(1, dtype=torch.int32, device=dev)
    st = N.lib().qmoe_moe_align(c_void_p(topk_ids.data_ptr()), M, k, E, block, c_void_p(sorted_ids.data_ptr()),
                                c_void_p(expert_ids.data_ptr()), c_void_p(npp.data_ptr()), capacity,
                                _stream_ptr(stream))
    N.check(st, "qmoe_moe_align")
    return sorted_ids[:capacity], expert_ids[:-(-capacity // block)], npp


def qmoe_workspace_size(layer: DeviceLayer, M: int, k: int, opts=None) -> int:
    if opts is None:
        n = N.lib().qmoe_workspace_size(byref(layer.struct), M, k)
    else:
        n = N.lib().qmoe_workspace_size_ex(byref(layer.struct), M, k, byref(opts))
    if n == 0 and M > 0:
        raise N.QmoeError(N.QMOE_ERR_INVALID_ARG, "qmoe_workspace_size")
    return int(n)


def qmoe_describe_plan(layer, M: int, k: int, opts=None, num_sms: int = 0) -> dict:
    """The launch plan of a forward (token tile, issuers, splits, ring depths,
    workspace bytes) for a DeviceLayer or a raw QmoeLayer struct; host only
    when num_sms > 0."""
    struct = layer.struct if hasattr(layer, "struct") else layer
    info = N.QmoePlanInfo()
    st = N.lib().qmoe_describe_plan(byref(struct), M, k, None if opts is None else byref(opts), num_sms, byref(info))
    N.check(st, "qmoe_describe_plan")
    return {f: getattr(info, f) for f, _ in N.QmoePlanInfo._fields_ if f != "reserved"}


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def qmoe_forward(layer: DeviceLayer, x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                 out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, opts=None, stream=None):
    M, H = x.shape
    k = topk_ids.shape[1]
    assert x.dtype == layer.torch_dtype and x.is_contiguous() and H == layer.H
    assert topk_ids.dtype == torch.int32 and topk_weights.dtype == torch.float32
    assert topk_ids.is_contiguous() and topk_weights.is_contiguous()
    if out is None:
        out = torch.empty_like(x)
    if workspace is None:
        workspace = alloc_workspace(qmoe_workspace_size(layer, M, k, opts), x.device)
    args = (byref(layer.struct), c_void_p(x.data_ptr()), M, c_void_p(topk_ids.data_ptr()),
            c_void_p(topk_weights.data_ptr()), k, c_void_p(out.data_ptr()), c_void_p(workspace.data_ptr()),
            workspace.numel(), _stream_ptr(stream))
    if opts is None:
        st = N.lib().qmoe_forward(*args)
    else:
        st = N.lib().qmoe_forward_ex(*args, byref(opts))
    N.check(st, "qmoe_forward")
    return out


def qmoe_forward_profiled(layer: DeviceLayer, x, topk_ids, topk_weights, out, workspace, events, opts=None,
                          stream=None) -> int:
    """qmoe_forward_ex with the 14 torch.cuda.Event objects recorded around its seven launch slots
    (see include/qmoe.h).  Returns the number of kernels launched."""
    from ctypes import c_int32 as _i32
    M = x.shape[0]
    k = topk_ids.shape[1]
    for e in events:
        if e.cuda_event == 0:  # torch creates the CUDA event on its first record
            e.record(torch.cuda.current_stream() if stream is None else stream)
    evs = (c_void_p * len(events))(*[c_void_p(e.cuda_event) for e in events])
    n = _i32(0)
    st = N.lib().qmoe_forward_profiled(byref(layer.struct), c_void_p(x.data_ptr()), M, c_void_p(topk_ids.data_ptr()),
                                       c_void_p(topk_weights.data_ptr()), k, c_void_p(out.data_ptr()),
                                       c_void_p(workspace.data_ptr()), workspace.numel(), _stream_ptr(stream),
                                       None if opts is None else byref(opts), evs, len(events), byref(n))
    N.check(st, "qmoe_forward_profiled")
    return int(n.value)


def qmoe_workspace_size_host(layer: DeviceLayer, M: int, k: int) -> int:
    return int(N.lib().qmoe_workspace_size_host(byref(layer.struct), M, k))


def qmoe_forward_host(layer: DeviceLayer, x_host: torch.Tensor, topk_ids_host: torch.Tensor,
                      topk_weights_host: torch.Tensor, out_host: torch.Tensor, workspace: torch.Tensor, stream=None):
    """Host buffers in and out (pinned recommended); returns once the work is enqueued."""
    M, _ = x_host.shape
    k = topk_ids_host.shape[1]
    st = N.lib().qmoe_forward_host(byref(layer.struct), c_void_p(x_host.data_ptr()), M,
                                   c_void_p(topk_ids_host.data_ptr()), c_void_p(topk_weights_host.data_ptr()), k,
                                   c_void_p(out_host.data_ptr()), c_void_p(workspace.data_ptr()), workspace.numel(),
                                   _stream_ptr(stream))
    N.check(st, "qmoe_forward_host")
    return out_host


def qmoe_read_device_status(workspace: torch.Tensor, stream=None) -> int:
    return int(N.lib().qmoe_read_device_status(c_void_p(workspace.data_ptr()), _stream_ptr(stream)))


def qmoe_forward_noalloc(layer: DeviceLayer, x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                         out: torch.Tensor | None = None, stream=None):
    """qmoe_forward with the library's built-in 64 MiB device scratch instead of a
    caller workspace, for callers that may not allocate (see include/qmoe.h)."""
    M = x.shape[0]
    k = topk_ids.shape[1]
    if out is None:
        out = torch.empty_like(x)
    st = N.lib().qmoe_forward_noalloc(byref(layer.struct), c_void_p(x.data_ptr()), M, c_void_p(topk_ids.data_ptr()),
                                      c_void_p(topk_weights.data_ptr()), k, c_void_p(out.data_ptr()),
                                      _stream_ptr(stream))
    N.check(st, "qmoe_forward_noalloc")
    return out


def qmoe_read_noalloc_status(stream=None) -> int:
    """Device-side fault recorded by the last qmoe_forward_noalloc on the current device."""
    return int(N.lib().qmoe_read_noalloc_status(_stream_ptr(stream)))


_LOGIT_DT = {torch.float32: N.QMOE_F32, torch.float16: N.QMOE_F16, torch.bfloat16: N.QMOE_BF16}


def qmoe_route_topk(logits: torch.Tensor, k: int, renormalize: bool = True, topk_ids: torch.Tensor | None = None,
                    topk_weights: torch.Tensor | None = None, stream=None):
    """Top-k router on the GPU (softmax, top-k with ties to the lower id,
    optional renormalisation): returns (topk_ids int32 [M, k], topk_weights float32 [M, k])."""
    assert logits.is_cuda and logits.is_contiguous() and logits.dim() == 2 and logits.dtype in _LOGIT_DT
    M, E = logits.shape
    if topk_ids is None:
        topk_ids = torch.empty((M, k), dtype=torch.int32, device=logits.device)
    if topk_weights is None:
        topk_weights = torch.empty((M, k), dtype=torch.float32, device=logits.device)
    st = N.lib().qmoe_route_topk(c_void_p(logits.data_ptr()), _LOGIT_DT[logits.dtype], M, E, k,
                                 1 if renormalize else 0, c_void_p(topk_ids.data_ptr()),
                                 c_void_p(topk_weights.data_ptr()), _stream_ptr(stream))
    N.check(st, "qmoe_route_topk")
    return topk_ids, topk_weights


def qmoe_workspace_size_logits(layer: DeviceLayer, M: int, k: int) -> int:
    n = int(N.lib().qmoe_workspace_size_logits(byref(layer.struct), M, k))
    if n == 0:
        raise N.QmoeError(N.QMOE_ERR_INVALID_ARG, "qmoe_workspace_size_logits")
    return n


def qmoe_forward_logits(layer: DeviceLayer, x: torch.Tensor, logits: torch.Tensor, k: int, renormalize: bool = True,
                        out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None):
    """The router then the layer in one call (routing kept in the workspace)."""
    M, H = x.shape
    assert x.dtype == layer.torch_dtype and x.is_contiguous() and H == layer.H
    assert logits.is_contiguous() and logits.shape == (M, layer.E) and logits.dtype in _LOGIT_DT
    if out is None:
        out = torch.empty_like(x)
    if workspace is None:
        workspace = alloc_workspace(qmoe_workspace_size_logits(layer, M, k), x.device)
    st = N.lib().qmoe_forward_logits(byref(layer.struct), c_void_p(x.data_ptr()), M, c_void_p(logits.data_ptr()),
                                     _LOGIT_DT[logits.dtype], k, 1 if renormalize else 0, c_void_p(out.data_ptr()),
                                     c_void_p(workspace.data_ptr()), workspace.numel(), _stream_ptr(stream))
    N.check(st, "qmoe_forward_logits")
    return out


# ----------------------------------------------------------------------------
# dense linear layer
# ----------------------------------------------------------------------------
class DeviceLinear:
    """One packed [N, K] weight matrix on a CUDA device plus its C descriptor."""

    def __init__(self, qt, N_out, K, act, w, s=None, perm=None, group_size=None):
        self.qt, self.N, self.K, self.act = qt, N_out, K, act
        self.group_size = default_group_size(qt) if group_size is None else group_size
        self.w, self.s, self.perm = w, s, perm
        self.struct = N.QmoeLinear(N_out, K, self.group_size, _QT[qt], _ACT[act],
                                   N.QMOE_F32 if _float_scales(qt, self.group_size) else _ACT[act], w.data_ptr(),
                                   None if s is None else s.data_ptr(), None if perm is None else perm.data_ptr())

    @property
    def torch_dtype(self):
        return _TORCH_ACT[self.act]

    @classmethod
    def from_canonical(cls, qt, act, q, s, group_size=None, z=None, g_idx=None, device="cuda"):
        """Pack canonical codes [N, K] and scales (see qmoe_pack_linear) and upload them."""
        N_out, K = q.shape
        gs = default_group_size(qt) if group_size is None else group_size
        pk = qmoe_pack_linear(qt, N_out, K, act, q, s, gs, z, g_idx)

        def dev(a):
            return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device)
        return cls(qt, N_out, K, act, dev(pk["w"]), dev(pk["s"]), dev(pk["perm"]), gs)


def qmoe_linear_workspace_size(layer: DeviceLinear, M: int, opts=None) -> int:
    n = int(N.lib().qmoe_linear_workspace_size(byref(layer.struct), M, None if opts is None else byref(opts)))
    if n == 0:
        raise N.QmoeError(N.QMOE_ERR_INVALID_ARG, "qmoe_linear_workspace_size")
    return n


def qmoe_linear_describe_plan(layer, M: int, opts=None, num_sms: int = 0) -> dict:
    struct = layer.struct if hasattr(layer, "struct") else layer
    info = N.QmoePlanInfo()
    st = N.lib().qmoe_linear_describe_plan(byref(struct), M, None if opts is None else byref(opts), num_sms,
                                           byref(info))
    N.check(st, "qmoe_linear_describe_plan")
    return {f: getattr(info, f) for f, _ in N.QmoePlanInfo._fields_ if f != "reserved"}


def qmoe_linear_forward(layer: DeviceLinear, x: torch.Tensor, out: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, opts=None, stream=None):
    """out[M, N] = x[M, K] . W^T on the GPU (the library's GEMM kernel)."""
    M, K = x.shape
    assert x.dtype == layer.torch_dtype and x.is_contiguous() and K == layer.K
    if out is None:
        out = torch.empty((M, layer.N), dtype=x.dtype, device=x.device)
    if workspace is None:
        workspace = alloc_workspace(qmoe_linear_workspace_size(layer, M, opts), x.device)
    st = N.lib().qmoe_linear_forward(byref(layer.struct), c_void_p(x.data_ptr()), M, c_void_p(out.data_ptr()),
                                     c_void_p(workspace.data_ptr()), workspace.numel(), _stream_ptr(stream),
                                     None if opts is None else byref(opts))
    N.check(st, "qmoe_linear_forward")
    return out
