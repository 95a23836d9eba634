"""Plain float64 CPU reference of the fused MoE layer with weight-only-quantized experts.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

What is computed, and where it comes from
-----------------------------------------
* Dequantization.  "Marlin moe integration" (description: GPTQ checkpoints
  ``gptq-4bit-128g`` with and without ``actorder_True``; review: the kernel
  receives INT4 weights and scales) gives int4 codes with one scale per group
  of 128 input channels, the group of channel k being ``g_idx[k]`` under
  act-order.  Zero point 8 (symmetric codes 0..15) is this build's reading;
  the pages print no formula.  "[Kernel] W8A16 Int8 inside FusedMoE"
  (feature description) gives symmetric per-column, per-expert int8 with the
  weights cast to the activation type before the matmul; a "column" is read
  as one output feature of the expert matrix.
* Expert FFN.  Mixtral-style experts: ``W13`` stacks the gate rows (0..I-1)
  over the up rows (I..2I-1); ``t = SiLU(gate·x) * (up·x)``, ``y = W2·t``.
  The pages name the Mixtral models and the fused MoE kernel but print no
  formula; this is the plain reading.
* Routing-weighted sum.  ``out[m] = sum_j topk_weights[m, j] * y(m, j)`` with
  ``y(m, j)`` the FFN of expert ``topk_ids[m, j]`` applied to token m.
* Router (the step before the layer; the pages are silent on it).  The
  Mixtral-style layers these kernels serve route each token by a softmax over
  its expert logits, keep the top-k experts, and renormalise the kept
  probabilities to sum to one (optionally not, as some many-expert models
  do).  Readings: experts are ranked by logit, ties go to the lower expert
  id, the slots are filled in rank order.
* moe_align_block_size.  "Marlin moe integration" (review thread: the
  ``moe_align_block_size_kernel`` the fused kernel relies on; block size 16
  tied to the Marlin tile) groups the token-expert pairs by expert and pads
  each expert's group to a multiple of the block size.  Readings for what the
  pages leave open: pair index p = m*k + j; within an expert pairs keep
  ascending p; padding and the tail hold the sentinel P; experts are laid out
  in ascending id; an expert with no pairs takes no block; blocks past the
  padded total map to expert -1; pairs whose id is outside [0, E) are dropped.

Everything is float64 (the oracle does not round intermediates); dequantized
weights are exact in float64 because codes have at most 8 bits and scales at
most 24.

Pins (CPU tests, none of which reuses these formulas): quantize/dequantize
round trip against the offline quantizer; act-order identity and joint
permutation invariance; closed-form layers built from scaled permutation
matrices; zero input and all-zero-point weights; linearity in the routing
weights and invariance under permuting the top-k slots; a scalar brute-force
layer on tiny inputs; moe_align against hand-worked examples, a brute-force
stable sort and its structural invariants.
"""
from __future__ import annotations

import math

import numpy as np


# ----------------------------------------------------------------------------
# dequantization
# ----------------------------------------------------------------------------
def dequant_int4(q: np.ndarray, s: np.ndarray, g_idx: np.ndarray | None,
                 group_size: int, zeros: np.ndarray | None = None) -> np.ndarray:
    """W[n, k] = (q[n, k] - z[g(k), n]) * s[g(k), n], float64 [N, K].

    q: codes 0..15 [N, K]; s: scales [K/G, N]; g(k) = g_idx[k] under
    act-order, else k // G ("Marlin moe integration": GPTQ 4-bit group-128,
    with or without act order); group_size -1 is one group over all of K
    (channel-wise, "Add GPTQ Marlin 2:4 sparse structured support" lists
    group 128 or -1).  z: per-group zero points [K/G, N] (asymmetric, AWQ
    style: "[WIP] AWQ Faster Kernels"), or 8 for every group when None.
    """
    N, K = q.shape
    if g_idx is None:
        g = np.arange(K) // (K if group_size < 0 else group_size)
    else:
        g = np.asarray(g_idx, np.int64)
    scale_nk = np.asarray(s, np.float64)[g, :].T          # [N, K]: s[g(k), n]
    zero_nk = 8.0 if zeros is None else np.asarray(zeros, np.float64)[g, :].T
    return (q.astype(np.float64) - zero_nk) * scale_nk


def decompress_24(values: np.ndarray, positions: np.ndarray, zero_code: int = 8) -> np.ndarray:
    """Dense codes [N, K] of a 2:4-compressed matrix ("Add GPTQ Marlin 2:4
    sparse structured support"): for every aligned group j of 4 input channels,
    values[n, 2j] and values[n, 2j+1] are the codes at channels 4j + i0 and
    4j + i1 with positions[n, j] = (i0, i1), i0 < i1; the other two channels
    hold `zero_code` (value 0: 8 for int4 codes with zero point 8, 0 for
    signed int8 codes).
    values: uint8 [N, K/2] (int4 codes) or int8 [N, K/2]; positions: int [N, K/4, 2]."""
    values = np.asarray(values)
    positions = np.asarray(positions, np.int64)
    N, half = values.shape
    K = 2 * half
    q = np.full((N, K), zero_code, values.dtype)
    rows = np.arange(N)[:, None]
    base = 4 * np.arange(K // 4)[None, :]
    q[rows, base + positions[:, :, 0]] = values[:, 0::2]
    q[rows, base + positions[:, :, 1]] = values[:, 1::2]
    return q


def dequant_int8(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """W[n, k] = q[n, k] * s[n] ("[Kernel] W8A16 Int8 inside FusedMoE": symmetric
    per-column, per-expert int8), float64 [N, K]."""
    return q.astype(np.float64) * np.asarray(s, np.float64)[:, None]


def dequant_int8_group(q: np.ndarray, s: np.ndarray, group_size: int) -> np.ndarray:
    """W[n, k] = q[n, k] * s[k // G, n]: symmetric int8 with one scale per group of
    G input channels ("Add GPTQ Marlin 2:4 sparse structured support" lists
    8-bit with group 128), float64 [N, K]."""
    K = q.shape[1]
    scale_nk = np.asarray(s, np.float64)[np.arange(K) // group_size, :].T
    return q.astype(np.float64) * scale_nk


def dequant_layer_expert(layer, e: int):
    """Dequantized (W13_e [2I, H], W2_e [H, I]) of expert e of a canonical layer."""
    wl = layer.wl
    if wl.qt in ("int4", "int4zp", "int4s24"):
        # int4s24: the canonical codes are dense, 8 (value 0) at the pruned channels
        g13 = None if layer.g13 is None else layer.g13[e]
        g2 = None if layer.g2 is None else layer.g2[e]
        z13 = None if layer.z13 is None else layer.z13[e]
        z2 = None if layer.z2 is None else layer.z2[e]
        w13 = dequant_int4(layer.q13[e], layer.s13[e], g13, wl.group_size, z13)
        w2 = dequant_int4(layer.q2[e], layer.s2[e], g2, wl.group_size, z2)
    elif wl.qt == "int8g" or (wl.qt == "int8s24" and wl.group_size > 0):
        # int8s24: the canonical codes are dense, 0 at the pruned channels
        w13 = dequant_int8_group(layer.q13[e], layer.s13[e], wl.group_size)
        w2 = dequant_int8_group(layer.q2[e], layer.s2[e], wl.group_size)
    else:
        w13 = dequant_int8(layer.q13[e], layer.s13[e])
        w2 = dequant_int8(layer.q2[e], layer.s2[e])
    return w13, w2


def dequant_linear(lin) -> np.ndarray:
    """Dequantized W [N, K] of a canonical dense linear layer (any format above)."""
    if lin.qt in ("int4", "int4zp", "int4s24"):
        return dequant_int4(lin.q, lin.s, lin.g_idx, lin.group_size, lin.z)
    if lin.qt == "int8g" or (lin.qt == "int8s24" and lin.group_size > 0):
        return dequant_int8_group(lin.q, lin.s, lin.group_size)
    return dequant_int8(lin.q, lin.s)


def linear_forward(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """out[m, n] = sum_k x[m, k] * W[n, k]: the dense linear layer that "Add GPTQ
    Marlin 2:4 sparse structured support" runs with 4- or 8-bit weights, dense
    or 2:4 sparse (float64)."""
    return np.asarray(x, np.float64) @ np.asarray(w, np.float64).T


# ----------------------------------------------------------------------------
# expert FFN and the routed layer
# ----------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z / (1 + exp(-z))."""
    return z / (1.0 + np.exp(-z))


def expert_ffn(xrows: np.ndarray, w13: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """y = W2 · (SiLU(gate·x) * (up·x)) for each row x of ``xrows`` [R, H]."""
    I = w13.shape[0] // 2
    h = np.asarray(xrows, np.float64) @ w13.T               # [R, 2I]
    t = silu(h[:, :I]) * h[:, I:]                           # [R, I]
    return t @ w2.T                                         # [R, H]


def moe_forward_batches(layer, batches, experts=None) -> list:
    """Layer outputs for the tokens ``rows`` of several token batches of one layer.

    batches: sequence of (x [M, H], topk_ids [M, k], topk_weights [M, k], rows).
    Returns one float64 [len(rows), H] array per batch (each token row is
    independent of the others).  Each expert's matrices are dequantized once
    for all batches.  With ``experts`` (a subset of expert ids) only the slots
    routed to those experts contribute: out[m] = sum over slots j with
    topk_ids[m, j] in ``experts`` of topk_weights[m, j] * y(m, j); summed over
    a partition of the experts this is the whole output.
    """
    E = layer.wl.E
    H = layer.wl.H
    todo = range(E) if experts is None else experts
    prep = []
    for x, topk_ids, topk_weights, rows in batches:
        rows = np.asarray(list(rows), np.int64)
        ids = np.asarray(topk_ids)[rows]                    # [R, k]
        w = np.asarray(topk_weights, np.float64)[rows]      # [R, k]
        y = np.zeros((rows.size, ids.shape[1], H), np.float64)   # y(m, j); 0 for slots not computed
        prep.append((np.asarray(x, np.float64)[rows], ids, w, y))
    for e in todo:
        sels = [np.nonzero(ids == e) for _, ids, _, _ in prep]
        if all(sel[0].size == 0 for sel in sels):
            continue
        w13, w2 = dequant_layer_expert(layer, e)
        for (xr, _, _, y), sel in zip(prep, sels):
            if sel[0].size:
                y[sel[0], sel[1], :] = expert_ffn(xr[sel[0]], w13, w2)
        del w13, w2
    outs = []
    for _, ids, w, y in prep:
        out = np.zeros((ids.shape[0], H), np.float64)
        for j in range(ids.shape[1]):
            out += w[:, j:j + 1] * y[:, j, :]
        outs.append(out)
    return outs


def moe_forward_rows(layer, x: np.ndarray, topk_ids: np.ndarray,
                     topk_weights: np.ndarray, rows) -> np.ndarray:
    """Layer output for the tokens ``rows`` only (each row is independent).

    Returns float64 [len(rows), H].  Used to check sampled tokens of large
    workloads; ``moe_forward`` is this over all rows.
    """
    return moe_forward_batches(layer, [(x, topk_ids, topk_weights, rows)])[0]


def moe_forward(layer, x: np.ndarray, topk_ids: np.ndarray,
                topk_weights: np.ndarray) -> np.ndarray:
    """out[m] = sum_j topk_weights[m, j] * FFN_{topk_ids[m, j]}(x[m]), float64 [M, H]."""
    return moe_forward_rows(layer, x, topk_ids, topk_weights, range(np.asarray(x).shape[0]))


# ----------------------------------------------------------------------------
# router: softmax -> top-k -> (optional) renormalisation
# ----------------------------------------------------------------------------
def route_topk(logits: np.ndarray, k: int, renormalize: bool = True):
    """Top-k routing of each token row of ``logits`` [M, E].

    k rounds per row, each taking the largest logit not yet taken (the lowest
    expert id among equal logits).  Weights are the softmax probabilities of
    the kept experts, p_e = exp(l_e) / sum_j exp(l_j), divided by their sum
    when ``renormalize``; a row whose logits are all -inf routes uniformly.
    NaN logits count as -inf.  Returns (ids int32 [M, k], weights float64 [M, k]).
    """
    lg = np.asarray(logits, np.float64)
    lg = np.where(np.isnan(lg), -np.inf, lg)
    M, E = lg.shape
    ids = np.zeros((M, k), np.int32)
    w = np.zeros((M, k), np.float64)
    for m in range(M):
        row = lg[m]
        taken = np.zeros(E, bool)
        for r in range(k):
            best = -1
            for e in range(E):
                if taken[e]:
                    continue
                if best < 0 or row[e] > row[best]:
                    best = e
            taken[best] = True
            ids[m, r] = best
        top = row.max()
        # softmax numerators with the maximum shifted to 1 (a row of -inf logits: uniform)
        p = np.ones(E) if top == -np.inf else np.exp(row - top)
        kept = p[ids[m]]
        w[m] = kept / (kept.sum() if renormalize else p.sum())
    return ids, w


# ----------------------------------------------------------------------------
# moe_align_block_size
# ----------------------------------------------------------------------------
def moe_align(topk_ids: np.ndarray, E: int, block: int, capacity: int | None = None):
    """Group token-expert pairs by expert, padded per expert to ``block``.

    Returns (sorted_ids int32 [capacity], expert_ids int32 [ceil(capacity/block)],
    num_post_padded int).  Default capacity is the worst case P + E*(block-1).
    """
    flat = np.asarray(topk_ids).reshape(-1).astype(np.int64)
    P = flat.size
    if capacity is None:
        capacity = P + E * (block - 1)
    counts = [int(np.count_nonzero(flat == e)) for e in range(E)]
    padded = [int(math.ceil(c / block)) * block for c in counts]
    offsets = [0] * E
    for e in range(1, E):
        offsets[e] = offsets[e - 1] + padded[e - 1]
    total = sum(padded)
    sorted_ids = np.full(capacity, P, np.int32)
    expert_ids = np.full(-(-capacity // block), -1, np.int32)
    for e in range(E):
        pairs = np.nonzero(flat == e)[0]                    # ascending pair index
        sorted_ids[offsets[e]:offsets[e] + pairs.size] = pairs
        expert_ids[offsets[e] // block:(offsets[e] + padded[e]) // block] = e
    return sorted_ids, expert_ids, total
