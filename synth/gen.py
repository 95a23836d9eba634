"""Seeded generators for the layer's weights, activations and routing.

Shapes and value distributions follow the workloads the pages run the fused
MoE layer on (Mixtral-8x7B and 8x22B GPTQ int4 group-128 with and without
act-order, ExpertsInt8 per-column int8 on Mixtral and a DeepSeek-V2-like
many-expert layer).  Weights are N(0, 0.02) floats quantized offline by
round-to-nearest (the pages keep quantization off the kernel's path and in
test utilities), activations are N(0, 1), and router logits are N(0, 1)
(plus a Zipf(1.1) per-expert bias for the skewed many-expert layer), softmaxed
with top-k selection and renormalised.

Seeds: weights from ``seed`` (default 0), activations from ``seed + 1`` and
router logits from ``seed + 2``, each expert's matrices from their own
sub-stream so that generation can run in parallel and stays reproducible.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    name: str
    E: int            # experts
    k: int            # top-k
    H: int            # hidden size
    I: int            # expert intermediate size
    qt: str           # "int4" (zero point 8), "int4zp" (per-group zero points), "int4s24"
                      # (int4, 2:4 sparse along K), "int8" (per output column), "int8g"
                      # (group scales) or "int8s24" (int8, 2:4 sparse along K)
    group_size: int   # 128 or -1 (whole K is one group) for int4 / int4zp / int4s24 / int8s24;
                      # -1 for int8; 128 for int8g
    act: str          # activation / scale storage type: "f16" or "bf16"
    act_order: bool   # int4 only: random per-expert g_idx permutation
    zipf: float       # 0: unbiased router; >0: Zipf exponent of the per-expert logit bias
    Ms: tuple         # token counts this workload is measured at
    w_std: float = 0.02

    def flops(self, M: int) -> float:
        """Useful FLOPs of one layer call: 2·M·k·3·H·I (padding excluded)."""
        return 2.0 * M * self.k * 3.0 * self.H * self.I

    def expert_weight_bytes(self) -> int:
        """Stored weight + scale (+ zero point) bytes of one expert (W13 and W2)."""
        n = 3 * self.H * self.I
        groups = (2 * self.I + self.H) if self.group_size < 0 else n // self.group_size
        if self.qt == "int4":
            return n // 2 + groups * 2
        if self.qt == "int4s24":   # half the values, 2 bits of position each
            return n // 4 + n // 8 + groups * 2
        if self.qt == "int4zp":
            return n // 2 + groups * 2 + groups // 2
        if self.qt == "int8g":
            return n + groups * 2
        if self.qt == "int8s24":   # half the codes, 2 bits of position each
            return n // 2 + n // 8 + (groups * 2 if self.group_size > 0 else (2 * self.I + self.H) * 4)
        return n + (2 * self.I + self.H) * 4


WORKLOADS = {
    # small layer the oracle finishes in well under a second
    "tiny": Workload("tiny", 8, 2, 256, 512, "int4", 128, "f16", False, 0.0, (16,)),
    # Mixtral-8x7B GPTQ int4 g128 (decode sweep)
    "mixtral8x7b_w4": Workload("mixtral8x7b_w4", 8, 2, 4096, 14336, "int4", 128, "f16",
                               False, 0.0, (1, 4, 8, 16, 64)),
    # same shape with act-order g_idx
    "mixtral8x7b_w4_actorder": Workload("mixtral8x7b_w4_actorder", 8, 2, 4096, 14336, "int4",
                                        128, "f16", True, 0.0, (1, 16, 128, 512)),
    # same shape, ExpertsInt8 (per-column int8, bf16 activations)
    "mixtral8x7b_w8": Workload("mixtral8x7b_w8", 8, 2, 4096, 14336, "int8", -1, "bf16",
                               False, 0.0, (1, 16, 128, 512)),
    # DeepSeek-V2-like many-expert layer with a skewed router
    "deepseekv2_w8": Workload("deepseekv2_w8", 160, 6, 5120, 1536, "int8", -1, "bf16",
                              False, 1.1, (1, 32, 256, 1024)),
    # Mixtral-8x7B shape with 2:4-sparse int4 g128 experts
    "mixtral8x7b_w4s24": Workload("mixtral8x7b_w4s24", 8, 2, 4096, 14336, "int4s24", 128, "f16",
                                  False, 0.0, (1, 16, 64)),
    # Mixtral-8x7B shape with 2:4-sparse per-column int8 experts (bf16 activations)
    "mixtral8x7b_w8s24": Workload("mixtral8x7b_w8s24", 8, 2, 4096, 14336, "int8s24", -1, "bf16",
                                  False, 0.0, (1, 16, 64)),
    # Mixtral-8x22B prefill, tensor-core-bound
    "mixtral8x22b_w4": Workload("mixtral8x22b_w4", 8, 2, 6144, 16384, "int4", 128, "bf16",
                                False, 0.0, (2048, 4096, 8192)),
}


# ----------------------------------------------------------------------------
# storage rounding (float32 arrays holding values exact in the target type)
# ----------------------------------------------------------------------------
def round_to_f16(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, np.float32).astype(np.float16).astype(np.float32)


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bfloat16, returned as float32."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def round_to(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return round_to_f16(a)
    if dtype == "bf16":
        return round_to_bf16(a)
    if dtype == "f32":
        return np.asarray(a, np.float32)
    raise ValueError(dtype)


def to_u16_bits(a: np.ndarray, dtype: str) -> np.ndarray:
    """Bit patterns of float32 values that are exact in ``dtype`` (f16/bf16)."""
    a = np.ascontiguousarray(a, np.float32)
    if dtype == "f16":
        return a.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------
# offline round-to-nearest quantizers (test utilities, not the kernel path)
# ----------------------------------------------------------------------------
def quantize_int4_rtn(w: np.ndarray, group_size: int, g_idx: np.ndarray | None,
                      scale_dtype: str):
    """Symmetric int4 with zero point 8 and one scale per (group, output row).

    w: float32 [N, K]; g_idx: int32 [K] group of each input channel (None:
    channel k is in group k // group_size).  Returns codes uint8 [N, K] in
    0..15 and scales float32 [K/G, N] holding values exact in ``scale_dtype``.
    Scale = absmax/7 of the group (a zero group gets scale 1), rounded to the
    storage type; codes = clamp(rint(w/scale), -8, 7) + 8.
    """
    N, K = w.shape
    G = K if group_size < 0 else group_size
    ng = K // G
    if g_idx is None:
        g_idx = (np.arange(K) // G).astype(np.int32)
    order = np.argsort(g_idx, kind="stable")
    grouped = np.abs(w[:, order]).reshape(N, ng, G)
    absmax = grouped.max(axis=2)                      # [N, ng]
    s = absmax / np.float32(7.0)
    s[s == 0] = 1.0
    s = round_to(s, scale_dtype).astype(np.float32)   # [N, ng]
    s_el = s[:, g_idx]                                # [N, K]
    q = np.clip(np.rint(w / s_el), -8, 7) + 8
    return q.astype(np.uint8), np.ascontiguousarray(s.T)


def prune_24(w: np.ndarray) -> np.ndarray:
    """2:4 structured sparsity along K: in every aligned group of 4 input
    channels keep the 2 entries of largest magnitude (ties go to the lower
    channel) and zero the other 2.  w: float32 [N, K], K % 4 == 0."""
    N, K = w.shape
    g = np.abs(w).reshape(N, K // 4, 4)
    # stable descending order by magnitude: lower index first among equals
    order = np.argsort(-g, axis=2, kind="stable")
    keep = np.zeros_like(g, dtype=bool)
    np.put_along_axis(keep, order[:, :, :2], True, axis=2)
    return np.where(keep.reshape(N, K), w, np.float32(0.0)).astype(np.float32)


def quantize_int4_24(w: np.ndarray, group_size: int, scale_dtype: str):
    """2:4-sparse int4 ("Add GPTQ Marlin 2:4 sparse structured support": 4-bit,
    group 128 or channel-wise): prune_24, then symmetric int4 RTN with zero
    point 8 on the pruned matrix, so every pruned entry has code 8 (value 0)
    and every aligned group of 4 codes along K holds at most 2 codes other
    than 8.  Returns codes uint8 [N, K] and scales float32 [K/G, N]."""
    return quantize_int4_rtn(prune_24(w), group_size, None, scale_dtype)


def quantize_int8_24(w: np.ndarray, group_size: int, scale_dtype: str):
    """2:4-sparse int8 ("Add GPTQ Marlin 2:4 sparse structured support": 8-bit,
    group 128 or channel-wise): prune_24, then symmetric int8 RTN on the pruned
    matrix (per output feature for group_size -1, per 128 input channels
    otherwise), so every pruned entry has code 0 and every aligned group of 4
    codes along K holds at most 2 non-zero codes.  Returns codes int8 [N, K] and
    scales float32 [N] (channel-wise) or [K/G, N] (grouped)."""
    wp = prune_24(w)
    if group_size < 0:
        return quantize_int8_rtn(wp)
    return quantize_int8_group(wp, group_size, scale_dtype)


def quantize_int4_rtn_zp(w: np.ndarray, group_size: int, g_idx: np.ndarray | None, scale_dtype: str):
    """Asymmetric int4 (AWQ-style): one scale and one zero point per (group, output row).

    Scale = (max - min)/15 of the group (a constant group gets scale 1), rounded
    to the storage type; zero point z = clamp(rint(-min/scale), 0, 15); codes =
    clamp(rint(w/scale) + z, 0, 15).  Returns codes uint8 [N, K], scales float32
    [K/G, N] and zero points uint8 [K/G, N].
    """
    N, K = w.shape
    G = K if group_size < 0 else group_size
    ng = K // G
    if g_idx is None:
        g_idx = (np.arange(K) // G).astype(np.int32)
    order = np.argsort(g_idx, kind="stable")
    grouped = w[:, order].reshape(N, ng, G)
    lo = grouped.min(axis=2)
    hi = grouped.max(axis=2)
    s = (hi - lo) / np.float32(15.0)
    s[s == 0] = 1.0
    s = round_to(s, scale_dtype).astype(np.float32)
    z = np.clip(np.rint(-lo / s), 0, 15).astype(np.float32)
    q = np.clip(np.rint(w / s[:, g_idx]) + z[:, g_idx], 0, 15)
    return q.astype(np.uint8), np.ascontiguousarray(s.T), np.ascontiguousarray(z.T.astype(np.uint8))


def quantize_int8_group(w: np.ndarray, group_size: int, scale_dtype: str):
    """Symmetric int8 with one scale per (group of input channels, output row):
    scale = absmax/127 rounded to the storage type, codes in -127..127.
    Returns codes int8 [N, K] and scales float32 [K/G, N]."""
    N, K = w.shape
    G = group_size
    absmax = np.abs(w).reshape(N, K // G, G).max(axis=2)
    s = absmax / np.float32(127.0)
    s[s == 0] = 1.0
    s = round_to(s, scale_dtype).astype(np.float32)
    q = np.clip(np.rint(w / np.repeat(s, G, axis=1)), -127, 127)
    return q.astype(np.int8), np.ascontiguousarray(s.T)


def quantize_int8_rtn(w: np.ndarray):
    """Symmetric per-output-column int8: scale = absmax/127 (float32), codes in -127..127."""
    absmax = np.abs(w).max(axis=1)
    s = (absmax / np.float32(127.0)).astype(np.float32)
    s[s == 0] = 1.0
    q = np.clip(np.rint(w / s[:, None]), -127, 127)
    return q.astype(np.int8), s


# ----------------------------------------------------------------------------
# layer weights
# ----------------------------------------------------------------------------
@dataclass
class QuantLayer:
    """Canonical (pre-pack) quantized expert weights.

    int4 / int4zp: q13 uint8 [E, 2I, H] (rows 0..I-1 gate, I..2I-1 up), s13
          float32 [E, H/G, 2I]; q2 uint8 [E, H, I], s2 float32 [E, I/G, H];
          g13 int32 [E, H] / g2 int32 [E, I] or None (no act-order); int4zp
          also z13 uint8 [E, H/G, 2I], z2 uint8 [E, I/G, H] (G = K when the
          group size is -1).
    int8: q13 int8 [E, 2I, H], s13 float32 [E, 2I]; q2 int8 [E, H, I],
          s2 float32 [E, H]; no g_idx.
    int8g: q13 int8 [E, 2I, H], s13 float32 [E, H/G, 2I]; q2 int8 [E, H, I],
          s2 float32 [E, I/G, H]; no g_idx.
    """
    wl: Workload
    q13: np.ndarray
    s13: np.ndarray
    q2: np.ndarray
    s2: np.ndarray
    g13: np.ndarray | None = None
    g2: np.ndarray | None = None
    z13: np.ndarray | None = None
    z2: np.ndarray | None = None
    meta: dict = field(default_factory=dict)


def _actorder_gidx(rng: np.random.Generator, K: int, G: int) -> np.ndarray:
    """Random act-order: channel perm[i] lands in group i // G."""
    perm = rng.permutation(K)
    g = np.empty(K, np.int32)
    g[perm] = (np.arange(K) // G).astype(np.int32)
    return g


def _gen_expert(wl: Workload, seed: int, e: int):
    out = {}
    for mat, (N, K) in (("13", (2 * wl.I, wl.H)), ("2", (wl.H, wl.I))):
        sub = 0 if mat == "13" else 1
        rng = np.random.default_rng([seed, e, sub])
        w = rng.standard_normal((N, K), dtype=np.float32)
        w *= np.float32(wl.w_std)
        if wl.qt == "int4s24":
            q, s = quantize_int4_24(w, wl.group_size, wl.act)
            out[mat] = (q, s, None, None)
        elif wl.qt == "int8s24":
            q, s = quantize_int8_24(w, wl.group_size, wl.act)
            out[mat] = (q, s, None, None)
        elif wl.qt in ("int4", "int4zp"):
            g = None
            if wl.act_order:
                g = _actorder_gidx(np.random.default_rng([seed, e, 2 + sub]), K, wl.group_size)
            if wl.qt == "int4":
                q, s = quantize_int4_rtn(w, wl.group_size, g, wl.act)
                out[mat] = (q, s, g, None)
            else:
                q, s, z = quantize_int4_rtn_zp(w, wl.group_size, g, wl.act)
                out[mat] = (q, s, g, z)
        elif wl.qt == "int8g":
            q, s = quantize_int8_group(w, wl.group_size, wl.act)
            out[mat] = (q, s, None, None)
        else:
            q, s = quantize_int8_rtn(w)
            out[mat] = (q, s, None, None)
        del w
    return out


def make_layer(wl: Workload, seed: int = 0, threads: int | None = None) -> QuantLayer:
    E, H, I = wl.E, wl.H, wl.I
    z13 = z2 = None
    if wl.qt in ("int4", "int4zp", "int4s24", "int8g") or (wl.qt == "int8s24" and wl.group_size > 0):
        n13 = 1 if wl.group_size < 0 else H // wl.group_size
        n2 = 1 if wl.group_size < 0 else I // wl.group_size
        cdt = np.int8 if wl.qt in ("int8g", "int8s24") else np.uint8
        q13 = np.empty((E, 2 * I, H), cdt)
        s13 = np.empty((E, n13, 2 * I), np.float32)
        q2 = np.empty((E, H, I), cdt)
        s2 = np.empty((E, n2, H), np.float32)
        if wl.qt == "int4zp":
            z13 = np.empty((E, n13, 2 * I), np.uint8)
            z2 = np.empty((E, n2, H), np.uint8)
    else:
        q13 = np.empty((E, 2 * I, H), np.int8)
        s13 = np.empty((E, 2 * I), np.float32)
        q2 = np.empty((E, H, I), np.int8)
        s2 = np.empty((E, H), np.float32)
    g13 = np.empty((E, H), np.int32) if wl.act_order else None
    g2 = np.empty((E, I), np.int32) if wl.act_order else None

    def one(e):
        r = _gen_expert(wl, seed, e)
        q13[e], s13[e], g, z = r["13"]
        if g13 is not None:
            g13[e] = g
        if z13 is not None:
            z13[e] = z
        q2[e], s2[e], g, z = r["2"]
        if g2 is not None:
            g2[e] = g
        if z2 is not None:
            z2[e] = z

    if threads is None:
        threads = max(1, min(8, os.cpu_count() or 1))
    big = 3 * H * I > (1 << 22)
    if threads > 1 and big and E > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(E)))
    else:
        for e in range(E):
            one(e)
    return QuantLayer(wl, q13, s13, q2, s2, g13, g2, z13, z2)


@dataclass
class QuantLinear:
    """Canonical (pre-pack) quantized weight of one dense linear layer W [N, K].

    q: codes [N, K] (uint8 0..15 for the int4 formats, int8 for the int8
    formats); s: scales float32 [K/G, N] (int4 formats, grouped int8 formats;
    [1, N] for channel-wise int4) or [N] (per-column int8 formats); z: zero
    points uint8 like s (int4zp); g_idx: int32 [K] act-order groups or None.
    """
    qt: str
    act: str
    group_size: int
    q: np.ndarray
    s: np.ndarray
    z: np.ndarray | None = None
    g_idx: np.ndarray | None = None


def make_linear(N: int, K: int, qt: str, group_size: int, act: str, act_order: bool = False, seed: int = 0,
                w_std: float = 0.02) -> QuantLinear:
    """A dense linear layer's weight, N(0, w_std) quantized offline like the experts."""
    rng = np.random.default_rng([seed, 7, 0])
    w = rng.standard_normal((N, K), dtype=np.float32)
    w *= np.float32(w_std)
    g = _actorder_gidx(np.random.default_rng([seed, 7, 1]), K, group_size) if act_order else None
    if qt == "int4":
        q, s = quantize_int4_rtn(w, group_size, g, act)
        return QuantLinear(qt, act, group_size, q, s, None, g)
    if qt == "int4zp":
        q, s, z = quantize_int4_rtn_zp(w, group_size, g, act)
        return QuantLinear(qt, act, group_size, q, s, z, g)
    if qt == "int4s24":
        q, s = quantize_int4_24(w, group_size, act)
        return QuantLinear(qt, act, group_size, q, s)
    if qt == "int8s24":
        q, s = quantize_int8_24(w, group_size, act)
        return QuantLinear(qt, act, group_size, q, s)
    if qt == "int8g":
        q, s = quantize_int8_group(w, group_size, act)
        return QuantLinear(qt, act, group_size, q, s)
    q, s = quantize_int8_rtn(w)
    return QuantLinear("int8", act, -1, q, s)


def make_linear_inputs(K: int, M: int, act: str, seed: int = 0) -> np.ndarray:
    """Activations [M, K] ~ N(0, 1), exact in the activation type."""
    return round_to(np.random.default_rng(seed + 1).standard_normal((M, K), dtype=np.float32), act)


# ----------------------------------------------------------------------------
# activations and routing
# ----------------------------------------------------------------------------
@dataclass
class Inputs:
    x: np.ndarray             # float32 [M, H], values exact in the activation type
    topk_ids: np.ndarray      # int32 [M, k]
    topk_weights: np.ndarray  # float32 [M, k]
    logits: np.ndarray        # float32 [M, E]


def route_topk(logits: np.ndarray, k: int):
    """Softmax -> top-k (ties go to the lower expert id) -> renormalise."""
    z = logits.astype(np.float64)
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    ids = np.argsort(-p, axis=1, kind="stable")[:, :k]
    w = np.take_along_axis(p, ids, axis=1)
    w /= w.sum(axis=1, keepdims=True)
    return ids.astype(np.int32), w.astype(np.float32)


def make_inputs(wl: Workload, M: int, seed: int = 0) -> Inputs:
    rx = np.random.default_rng(seed + 1)
    x = round_to(rx.standard_normal((M, wl.H), dtype=np.float32), wl.act)
    rr = np.random.default_rng(seed + 2)
    logits = rr.standard_normal((M, wl.E), dtype=np.float32)
    if wl.zipf > 0:
        rank = np.random.default_rng([seed + 2, 1]).permutation(wl.E) + 1
        logits = logits + (-wl.zipf * np.log(rank)).astype(np.float32)[None, :]
    ids, w = route_topk(logits, wl.k)
    return Inputs(x, ids, w, logits.astype(np.float32))
