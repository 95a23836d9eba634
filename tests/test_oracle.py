"""Pins for the CPU oracle (no GPU).

Each check ties the oracle to something other than its own formulas: the
offline quantizer it inverts, closed forms of layers built from scaled
permutation matrices, algebraic invariants of the routed sum, a scalar
brute-force layer, and hand-worked moe_align examples.  A plausible slip in
the oracle (a dropped zero point, a transposed operand, SiLU on the wrong half,
a wrong scale or group index, a lost routing weight, an unstable sort) fails
at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from synth import (QuantLayer, Workload, make_inputs, make_layer, make_linear, make_linear_inputs, prune_24,
                   quantize_int4_24, quantize_int4_rtn, quantize_int4_rtn_zp, quantize_int8_24, quantize_int8_group,
                   quantize_int8_rtn)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _wl(**kw):
    base = dict(name="t", E=4, k=2, H=32, I=64, qt="int4", group_size=16, act="f16",
                act_order=False, zipf=0.0, Ms=(3,))
    base.update(kw)
    return Workload(**base)


# ----------------------------------------------------------------------------
# dequantization vs the offline quantizer
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("act_order", [False, True])
@pytest.mark.parametrize("sdt", ["f16", "bf16"])
def test_int4_round_trip(act_order, sdt):
    rng = np.random.default_rng(5)
    N, K, G = 48, 256, 32
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    g = None
    if act_order:
        perm = rng.permutation(K)
        g = np.empty(K, np.int32)
        g[perm] = np.arange(K) // G
    q, s = quantize_int4_rtn(w, G, g, sdt)
    assert q.dtype == np.uint8 and q.min() >= 0 and q.max() <= 15
    assert s.shape == (K // G, N)
    wh = oracle.dequant_int4(q, s, g, G)
    gk = (np.arange(K) // G) if g is None else g
    half_step = 0.5 * s[gk, :].T.astype(np.float64)
    err = np.abs(w.astype(np.float64) - wh)
    assert np.all(err <= half_step * (1 + 1e-5) + 1e-12)
    # the largest code of each group reaches the group's absmax within a step
    assert np.all(np.abs(wh).max(axis=1) > 0)


def test_int4_dequant_hand_values():
    # two rows, four channels, group size 2; scales are powers of two
    q = np.array([[8, 9, 0, 15], [7, 8, 12, 4]], np.uint8)
    s = np.array([[0.5, 0.25], [2.0, 1.0]], np.float32)      # [K/G, N]
    want = np.array([[0.0, 0.5, -16.0, 14.0], [-0.25, 0.0, 4.0, -4.0]])
    assert np.array_equal(oracle.dequant_int4(q, s, None, 2), want)
    # act-order: channels 0 and 3 in group 1, channels 1 and 2 in group 0
    g = np.array([1, 0, 0, 1], np.int32)
    want_ao = np.array([[0.0, 0.5, -4.0, 14.0], [-1.0, 0.0, 1.0, -4.0]])
    assert np.array_equal(oracle.dequant_int4(q, s, g, 2), want_ao)


def test_int8_round_trip_and_hand_values():
    rng = np.random.default_rng(6)
    w = (rng.standard_normal((40, 96)) * 0.02).astype(np.float32)
    q, s = quantize_int8_rtn(w)
    assert q.dtype == np.int8 and q.min() >= -127 and q.max() <= 127
    wh = oracle.dequant_int8(q, s)
    assert np.all(np.abs(w - wh) <= 0.5 * s[:, None] * (1 + 1e-5))
    q2 = np.array([[1, -2], [127, -127]], np.int8)
    s2 = np.array([0.5, 0.25], np.float32)
    assert np.array_equal(oracle.dequant_int8(q2, s2), np.array([[0.5, -1.0], [31.75, -31.75]]))


# ----------------------------------------------------------------------------
# closed forms: experts built from scaled permutation matrices
# ----------------------------------------------------------------------------
def _perm_layer(qt, E, H, G, act_order, seed):
    """Gate = diag(a), up = b·P1, down = c·P2 per expert, with a, b, c varying per row.

    Returns the canonical layer plus the per-expert (pi1, pi2, a, b, c) that
    define the closed form y_h = c_h · SiLU(a_j x_j) · b_j x_{pi1(j)}, j = pi2(h).
    """
    I = H
    rng = np.random.default_rng(seed)
    wl = _wl(E=E, H=H, I=I, qt=qt, group_size=G if qt == "int4" else -1, act_order=act_order)
    spec = []
    if qt == "int4":
        q13 = np.full((E, 2 * I, H), 8, np.uint8)
        q2 = np.full((E, H, I), 8, np.uint8)
        s13 = np.zeros((E, H // G, 2 * I), np.float32)
        s2 = np.zeros((E, I // G, H), np.float32)
        g13 = np.zeros((E, H), np.int32) if act_order else None
        g2 = np.zeros((E, I), np.int32) if act_order else None
    else:
        q13 = np.zeros((E, 2 * I, H), np.int8)
        q2 = np.zeros((E, H, I), np.int8)
        s13 = np.zeros((E, 2 * I), np.float32)
        s2 = np.zeros((E, H), np.float32)
        g13 = g2 = None
    for e in range(E):
        pi1 = rng.permutation(H)
        pi2 = rng.permutation(I)
        if qt == "int4":
            ga = np.arange(H) // G
            gb = np.arange(I) // G
            if act_order:
                p = rng.permutation(H); ga = np.empty(H, np.int64); ga[p] = np.arange(H) // G
                p = rng.permutation(I); gb = np.empty(I, np.int64); gb[p] = np.arange(I) // G
                g13[e] = ga
                g2[e] = gb
            # power-of-two scales that differ by group and by row
            s13[e] = 2.0 ** -(1 + (np.arange(H // G)[:, None] + np.arange(2 * I)[None, :]) % 4)
            s2[e] = 2.0 ** -(1 + (2 * np.arange(I // G)[:, None] + np.arange(H)[None, :]) % 3)
            da = rng.integers(1, 8, I)          # gate code offset from zero point
            db = rng.integers(-8, 8, I)
            dc = rng.integers(-8, 8, H)
            a = np.empty(I); b = np.empty(I); c = np.empty(H)
            for j in range(I):
                q13[e, j, j] = 8 + da[j]
                a[j] = da[j] * s13[e, ga[j], j]
                q13[e, I + j, pi1[j]] = 8 + db[j]
                b[j] = db[j] * s13[e, ga[pi1[j]], I + j]
            for h in range(H):
                q2[e, h, pi2[h]] = 8 + dc[h]
                c[h] = dc[h] * s2[e, gb[pi2[h]], h]
        else:
            s13[e] = 2.0 ** -(2 + np.arange(2 * I) % 5)
            s2[e] = 2.0 ** -(1 + np.arange(H) % 3)
            da = rng.integers(1, 128, I)
            db = rng.integers(-127, 128, I)
            dc = rng.integers(-127, 128, H)
            a = np.empty(I); b = np.empty(I); c = np.empty(H)
            for j in range(I):
                q13[e, j, j] = da[j]; a[j] = da[j] * s13[e, j]
                q13[e, I + j, pi1[j]] = db[j]; b[j] = db[j] * s13[e, I + j]
            for h in range(H):
                q2[e, h, pi2[h]] = dc[h]; c[h] = dc[h] * s2[e, h]
        spec.append((pi1, pi2, a, b, c))
    return QuantLayer(wl, q13, s13, q2, s2, g13, g2), spec


def _closed_form(spec, x, ids, w):
    M, H = x.shape
    out = np.zeros((M, H))
    for m in range(M):
        for jj in range(ids.shape[1]):
            pi1, pi2, a, b, c = spec[ids[m, jj]]
            for h in range(H):
                j = pi2[h]
                gate = a[j] * x[m, j]
                up = b[j] * x[m, pi1[j]]
                out[m, h] += w[m, jj] * c[h] * (gate / (1.0 + math.exp(-gate))) * up
    return out


@pytest.mark.parametrize("qt,act_order", [("int4", False), ("int4", True), ("int8", False)])
def test_closed_form_permutation_experts(qt, act_order):
    E, H = 4, 32
    layer, spec = _perm_layer(qt, E, H, 8, act_order, seed=11)
    rng = np.random.default_rng(12)
    M, k = 5, 2
    x = rng.standard_normal((M, H))
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(M)]).astype(np.int32)
    w = rng.random((M, k)).astype(np.float32)
    got = oracle.moe_forward(layer, x, ids, w)
    want = _closed_form(spec, x, ids, w.astype(np.float64))
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_topk_all_experts_uniform_is_dense_average():
    E, H = 4, 16
    layer, spec = _perm_layer("int4", E, H, 8, False, seed=13)
    x = np.random.default_rng(14).standard_normal((3, H))
    ids = np.tile(np.arange(E, dtype=np.int32), (3, 1))
    w = np.full((3, E), 1.0 / E)
    got = oracle.moe_forward(layer, x, ids, w)
    dense = sum(_closed_form(spec, x, np.full((3, 1), e, np.int32), np.ones((3, 1))) for e in range(E)) / E
    np.testing.assert_allclose(got, dense, rtol=1e-12, atol=1e-13)


def test_top1_weight1_is_single_expert():
    layer, spec = _perm_layer("int8", 3, 16, 8, False, seed=15)
    x = np.random.default_rng(16).standard_normal((4, 16))
    for e in range(3):
        ids = np.full((4, 1), e, np.int32)
        got = oracle.moe_forward(layer, x, ids, np.ones((4, 1), np.float32))
        pi1, pi2, a, b, c = spec[e]
        want = np.empty_like(x)
        for m in range(4):
            for h in range(16):
                j = pi2[h]
                g = a[j] * x[m, j]
                want[m, h] = c[h] * g / (1 + math.exp(-g)) * b[j] * x[m, pi1[j]]
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------
# special cases and invariants on random quantized layers
# ----------------------------------------------------------------------------
@pytest.fixture(scope="module")
def small():
    wl = _wl(E=6, k=2, H=64, I=96, group_size=32, act_order=True)
    layer = make_layer(wl, seed=3)
    inp = make_inputs(wl, 7, seed=3)
    return wl, layer, inp


def test_zero_input_gives_zero(small):
    wl, layer, inp = small
    out = oracle.moe_forward(layer, np.zeros_like(inp.x), inp.topk_ids, inp.topk_weights)
    assert np.all(out == 0.0)


def test_zero_point_codes_give_zero(small):
    wl, layer, inp = small
    flat = QuantLayer(wl, np.full_like(layer.q13, 8), layer.s13, layer.q2, layer.s2, layer.g13, layer.g2)
    out = oracle.moe_forward(flat, inp.x, inp.topk_ids, inp.topk_weights)
    assert np.all(out == 0.0)
    flat2 = QuantLayer(wl, layer.q13, layer.s13, np.full_like(layer.q2, 8), layer.s2, layer.g13, layer.g2)
    assert np.all(oracle.moe_forward(flat2, inp.x, inp.topk_ids, inp.topk_weights) == 0.0)


def test_linear_in_routing_weights(small):
    wl, layer, inp = small
    rng = np.random.default_rng(21)
    w1 = rng.random(inp.topk_weights.shape)
    w2 = rng.random(inp.topk_weights.shape)
    o1 = oracle.moe_forward(layer, inp.x, inp.topk_ids, w1)
    o2 = oracle.moe_forward(layer, inp.x, inp.topk_ids, w2)
    o12 = oracle.moe_forward(layer, inp.x, inp.topk_ids, w1 + 3.0 * w2)
    np.testing.assert_allclose(o12, o1 + 3.0 * o2, rtol=1e-11, atol=1e-12)


def test_slot_permutation_invariance(small):
    wl, layer, inp = small
    o = oracle.moe_forward(layer, inp.x, inp.topk_ids, inp.topk_weights)
    rev = oracle.moe_forward(layer, inp.x, inp.topk_ids[:, ::-1], inp.topk_weights[:, ::-1])
    np.testing.assert_allclose(rev, o, rtol=1e-12, atol=1e-13)


def test_duplicate_expert_in_a_row_is_summed(small):
    wl, layer, inp = small
    ids = np.repeat(inp.topk_ids[:, :1], 2, axis=1)
    w = inp.topk_weights.astype(np.float64)
    o = oracle.moe_forward(layer, inp.x, ids, w)
    single = oracle.moe_forward(layer, inp.x, ids[:, :1], (w[:, 0] + w[:, 1])[:, None])
    np.testing.assert_allclose(o, single, rtol=1e-12, atol=1e-13)


def test_actorder_identity_gidx_matches_plain_groups():
    wl = _wl(E=3, H=64, I=64, group_size=16)
    layer = make_layer(wl, seed=8)
    inp = make_inputs(wl, 4, seed=8)
    ident13 = np.tile((np.arange(64) // 16).astype(np.int32), (3, 1))
    ident2 = ident13.copy()
    ao = QuantLayer(wl, layer.q13, layer.s13, layer.q2, layer.s2, ident13, ident2)
    a = oracle.moe_forward(layer, inp.x, inp.topk_ids, inp.topk_weights)
    b = oracle.moe_forward(ao, inp.x, inp.topk_ids, inp.topk_weights)
    assert np.array_equal(a, b)


def test_actorder_joint_permutation_invariance(small):
    wl, layer, inp = small
    rng = np.random.default_rng(9)
    ph = rng.permutation(wl.H)      # hidden channels: x columns, W13 K dim, g13
    pi = rng.permutation(wl.I)      # intermediate channels: gate/up rows, W2 K dim, g2
    rows13 = np.concatenate([pi, wl.I + pi])
    L2 = QuantLayer(wl,
                    layer.q13[:, rows13][:, :, ph], layer.s13[:, :, rows13],
                    layer.q2[:, :, pi], layer.s2,
                    layer.g13[:, ph], layer.g2[:, pi])
    # the permuted W2 K order also moves the output rows of W13, so the output
    # columns of W2 (hidden) stay put while the input columns move with ph
    o = oracle.moe_forward(layer, inp.x, inp.topk_ids, inp.topk_weights)
    o2 = oracle.moe_forward(L2, inp.x[:, ph], inp.topk_ids, inp.topk_weights)
    np.testing.assert_allclose(o2, o, rtol=1e-11, atol=1e-12)


def _brute_force(layer, x, ids, w):
    """Scalar loops straight from the definitions, dequantizing inside the dot products."""
    wl = layer.wl
    E, H, I = wl.E, wl.H, wl.I
    M, k = ids.shape
    out = [[0.0] * H for _ in range(M)]

    def wq(q, s, gi, z, e, n, c):
        if wl.qt in ("int4", "int4zp", "int4s24", "int8g") or (wl.qt == "int8s24" and wl.group_size > 0):
            if gi is not None:
                g = int(gi[e, c])
            elif wl.group_size < 0:
                g = 0
            else:
                g = c // wl.group_size
            zero = 0 if wl.qt in ("int8g", "int8s24") else (8 if z is None else int(z[e, g, n]))
            return (int(q[e, n, c]) - zero) * float(s[e, g, n])
        return int(q[e, n, c]) * float(s[e, n])

    def wq13(e, n, c):
        return wq(layer.q13, layer.s13, layer.g13, layer.z13, e, n, c)

    def wq2(e, h, c):
        return wq(layer.q2, layer.s2, layer.g2, layer.z2, e, h, c)

    for m in range(M):
        for j in range(k):
            e = int(ids[m, j])
            t = []
            for i in range(I):
                gsum = 0.0
                usum = 0.0
                for c in range(H):
                    gsum += wq13(e, i, c) * float(x[m, c])
                    usum += wq13(e, I + i, c) * float(x[m, c])
                t.append(gsum / (1.0 + math.exp(-gsum)) * usum)
            for h in range(H):
                acc = 0.0
                for i in range(I):
                    acc += wq2(e, h, i) * t[i]
                out[m][h] += float(w[m, j]) * acc
    return np.array(out)


@pytest.mark.parametrize("qt,act_order,gs", [("int4", False, 16), ("int4", True, 16), ("int8", False, -1),
                                             ("int4zp", False, 16), ("int4zp", True, 16), ("int4", False, -1),
                                             ("int4zp", False, -1), ("int8g", False, 16), ("int4s24", False, 16),
                                             ("int4s24", False, -1), ("int8s24", False, -1), ("int8s24", False, 16)])
def test_brute_force_tiny(qt, act_order, gs):
    wl = _wl(E=4, k=2, H=32, I=48, qt=qt, group_size=gs, act_order=act_order)
    layer = make_layer(wl, seed=17)
    inp = make_inputs(wl, 3, seed=17)
    got = oracle.moe_forward(layer, inp.x, inp.topk_ids, inp.topk_weights)
    want = _brute_force(layer, inp.x, inp.topk_ids, inp.topk_weights)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


def test_forward_rows_match_full(small):
    wl, layer, inp = small
    full = oracle.moe_forward(layer, inp.x, inp.topk_ids, inp.topk_weights)
    part = oracle.moe_forward_rows(layer, inp.x, inp.topk_ids, inp.topk_weights, [5, 1])
    assert np.array_equal(part, full[[5, 1]])


def test_forward_batches_partition_and_brute_force():
    """Several token sets of one layer in one call: each equals the scalar brute
    force of its rows; summed over a partition of the experts the per-subset
    outputs give the whole output, and an expert subset that no slot uses
    contributes exactly zero."""
    wl = _wl(E=5, k=2, H=32, I=48, group_size=16, act_order=True)
    layer = make_layer(wl, seed=23)
    a = make_inputs(wl, 6, seed=1)
    b = make_inputs(wl, 4, seed=2)
    batches = [(a.x, a.topk_ids, a.topk_weights, [4, 0, 2]), (b.x, b.topk_ids, b.topk_weights, [3, 1])]
    got = oracle.moe_forward_batches(layer, batches)
    for (x, ids, w, rows), g in zip(batches, got):
        want = _brute_force(layer, x[rows], ids[rows], w[rows])
        np.testing.assert_allclose(g, want, rtol=1e-10, atol=1e-12)
    parts = [oracle.moe_forward_batches(layer, batches, experts=sub) for sub in ([0, 3], [1], [2, 4])]
    for i in range(2):
        np.testing.assert_allclose(sum(p[i] for p in parts), got[i], rtol=1e-12, atol=1e-14)
    used = set(np.concatenate([a.topk_ids[[4, 0, 2]].ravel(), b.topk_ids[[3, 1]].ravel()]).tolist())
    unused = [e for e in range(wl.E) if e not in used]
    if unused:
        for z in oracle.moe_forward_batches(layer, batches, experts=unused):
            assert np.all(z == 0.0)


# ----------------------------------------------------------------------------
# moe_align
# ----------------------------------------------------------------------------
def test_moe_align_golden():
    with open(os.path.join(GOLDEN, "moe_align_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        ids = np.array(c["topk_ids"], np.int32)
        s, ex, n = oracle.moe_align(ids, c["E"], c["block"])
        assert s.tolist() == c["sorted_ids"], c["name"]
        assert ex.tolist() == c["expert_ids"], c["name"]
        assert n == c["num_post_padded"], c["name"]


def _align_by_sorting(ids, E, B):
    """Independent construction: stable sort of valid pairs by (expert, pair)."""
    flat = [int(v) for v in np.asarray(ids).reshape(-1)]
    P = len(flat)
    cap = P + E * (B - 1)
    order = sorted((p for p in range(P) if 0 <= flat[p] < E), key=lambda p: (flat[p], p))
    sorted_ids, expert_ids = [], []
    pos = 0
    while pos < len(order):
        e = flat[order[pos]]
        grp = [p for p in order[pos:] if flat[p] == e]
        pos += len(grp)
        while len(grp) % B:
            grp.append(P)
        sorted_ids += grp
        expert_ids += [e] * (len(grp) // B)
    total = len(sorted_ids)
    sorted_ids += [P] * (cap - total)
    expert_ids += [-1] * (-(-cap // B) - len(expert_ids))
    return sorted_ids, expert_ids, total


@pytest.mark.parametrize("M,k,E,B", [(1, 2, 8, 16), (17, 2, 8, 16), (64, 6, 160, 16),
                                     (33, 2, 8, 64), (100, 4, 16, 1), (5, 8, 3, 4)])
def test_moe_align_vs_sort_and_invariants(M, k, E, B):
    rng = np.random.default_rng(M * 131 + E)
    ids = rng.integers(0, E, (M, k)).astype(np.int32)
    s, ex, n = oracle.moe_align(ids, E, B)
    rs, rex, rn = _align_by_sorting(ids, E, B)
    assert s.tolist() == rs and ex.tolist() == rex and n == rn
    P = M * k
    real = s[s < P]
    assert sorted(real.tolist()) == list(range(P))
    assert n % B == 0
    for b in range(n // B):
        blk = s[b * B:(b + 1) * B]
        e = ex[b]
        assert all(ids.reshape(-1)[p] == e for p in blk if p < P)
    assert np.all(ex[n // B:] == -1)


# ----------------------------------------------------------------------------
# router: softmax -> top-k -> renormalise
# ----------------------------------------------------------------------------
def test_route_topk_hand_examples():
    # ties go to the lower expert id, slots in rank order
    ids, w = oracle.route_topk(np.array([[1.0, 3.0, 3.0, 0.0]]), 2)
    assert ids.tolist() == [[1, 2]]
    np.testing.assert_allclose(w, [[0.5, 0.5]], rtol=0, atol=1e-15)
    # renormalised top-2 of logits (0, ln 3): weights 1/4 and 3/4, the larger first
    ids, w = oracle.route_topk(np.array([[0.0, math.log(3.0), -50.0]]), 2)
    assert ids.tolist() == [[1, 0]]
    np.testing.assert_allclose(w, [[0.75, 0.25]], rtol=1e-14)
    # without renormalisation the weights are the plain softmax probabilities
    ids, w = oracle.route_topk(np.array([[0.0, math.log(3.0), math.log(4.0)]]), 1, renormalize=False)
    assert ids.tolist() == [[2]]
    np.testing.assert_allclose(w, [[0.5]], rtol=1e-14)       # 4 / (1 + 3 + 4)


def test_route_topk_vs_sort_and_closed_forms():
    rng = np.random.default_rng(11)
    for E, k in [(8, 2), (16, 5), (160, 6), (7, 7)]:
        # integer-valued logits make ties frequent
        lg = rng.integers(-3, 4, size=(40, E)).astype(np.float64) * 0.5
        ids, w = oracle.route_topk(lg, k)
        idsn, wn = oracle.route_topk(lg, k, renormalize=False)
        for m in range(lg.shape[0]):
            want = sorted(range(E), key=lambda e: (-lg[m, e], e))[:k]   # stable rank order
            assert ids[m].tolist() == want and idsn[m].tolist() == want
            assert len(set(ids[m].tolist())) == k
            # renormalised weights: sum 1, ratios exp(l_i - l_j)
            assert abs(w[m].sum() - 1.0) < 1e-12
            for r in range(1, k):
                assert abs(w[m, r] / w[m, 0] - math.exp(lg[m, want[r]] - lg[m, want[0]])) < 1e-12
            # plain softmax: against the full distribution computed directly
            full = np.exp(lg[m]) / np.exp(lg[m]).sum()
            np.testing.assert_allclose(wn[m], full[want], rtol=1e-12)
        if k == E:
            assert np.allclose(wn.sum(axis=1), 1.0)


def test_route_topk_large_logits_do_not_overflow():
    lg = np.array([[1e4, 1e4 - 1.0, -1e4], [-1e4, -1e4 + math.log(2.0), 0.0]])
    ids, w = oracle.route_topk(lg, 2)
    assert ids.tolist() == [[0, 1], [2, 1]]
    np.testing.assert_allclose(w[0], [1 / (1 + math.exp(-1)), math.exp(-1) / (1 + math.exp(-1))], rtol=1e-12)
    np.testing.assert_allclose(w[1], [1.0, 0.0], atol=1e-12)


def test_route_topk_masked_rows():
    inf = math.inf
    ids, w = oracle.route_topk(np.array([[-inf, 2.0, -inf, float("nan")], [-inf] * 4]), 3)
    assert ids[0].tolist() == [1, 0, 2] and ids[1].tolist() == [0, 1, 2]
    np.testing.assert_allclose(w[0], [1.0, 0.0, 0.0])
    np.testing.assert_allclose(w[1], [1 / 3] * 3)
    _, wn = oracle.route_topk(np.array([[-inf] * 4]), 2, renormalize=False)
    np.testing.assert_allclose(wn[0], [0.25, 0.25])


# ----------------------------------------------------------------------------
# other weight formats: asymmetric int4 (zero points), channel-wise int4, grouped int8
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("act_order", [False, True])
@pytest.mark.parametrize("sdt", ["f16", "bf16"])
def test_int4_zero_point_round_trip(act_order, sdt):
    rng = np.random.default_rng(21)
    N, K, G = 24, 256, 128
    w = (rng.standard_normal((N, K)) * 0.02 + 0.01).astype(np.float32)   # off-centre groups
    g = None
    if act_order:
        perm = rng.permutation(K)
        g = np.empty(K, np.int32)
        g[perm] = np.arange(K) // G
    q, s, z = quantize_int4_rtn_zp(w, G, g, sdt)
    assert q.max() <= 15 and z.max() <= 15
    wd = oracle.dequant_int4(q, s, g, G, z)
    gk = (np.arange(K) // G) if g is None else g
    s_el = s[gk, :].T
    assert np.all(np.abs(wd - w) <= s_el * (1.0 + 1e-6))                 # within one step
    inside = (q > 0) & (q < 15)
    assert np.all(np.abs(wd - w)[inside] <= s_el[inside] * (0.5 + 1e-6))  # half a step unless clipped


def test_int4_zero_point_hand_values_and_symmetric_case():
    q = np.array([[3, 12, 0, 15]], np.uint8)
    s = np.array([[0.5, 0.25]])                 # [K/G, N] with G = 2, N = 1 -> shape [2, 1]
    s = s.T
    z = np.array([[5], [15]], np.uint8)
    got = oracle.dequant_int4(q, s, None, 2, z)
    np.testing.assert_array_equal(got, [[-1.0, 3.5, -3.75, 0.0]])
    # zero points of 8 everywhere are the symmetric format, bit for bit
    rng = np.random.default_rng(2)
    q = rng.integers(0, 16, size=(16, 256)).astype(np.uint8)
    s = rng.random((2, 16)) + 0.1
    assert np.array_equal(oracle.dequant_int4(q, s, None, 128, np.full((2, 16), 8, np.uint8)),
                          oracle.dequant_int4(q, s, None, 128))


def test_int4_channel_wise_is_one_group():
    rng = np.random.default_rng(3)
    q = rng.integers(0, 16, size=(8, 256)).astype(np.uint8)
    s1 = rng.random((1, 8)) + 0.1
    a = oracle.dequant_int4(q, s1, None, -1)
    b = oracle.dequant_int4(q, np.repeat(s1, 2, axis=0), None, 128)   # the same scale in both groups
    c = oracle.dequant_int4(q, s1, None, 256)
    assert np.array_equal(a, b) and np.array_equal(a, c)
    w = rng.standard_normal((8, 256)).astype(np.float32) * 0.02
    qq, ss = quantize_int4_rtn(w, -1, None, "f16")
    assert ss.shape == (1, 8)
    assert np.all(np.abs(oracle.dequant_int4(qq, ss, None, -1) - w) <= ss[0][:, None] * (0.5 + 1e-6))


@pytest.mark.parametrize("sdt", ["f16", "bf16"])
def test_int8_group_round_trip_hand_values_and_per_column_case(sdt):
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((16, 384)) * 0.02).astype(np.float32)
    q, s = quantize_int8_group(w, 128, sdt)
    assert s.shape == (3, 16) and np.abs(q.astype(np.int32)).max() <= 127
    wd = oracle.dequant_int8_group(q, s, 128)
    assert np.all(np.abs(wd - w) <= np.repeat(s.T, 128, axis=1) * (0.5 + 1e-6))
    qh = np.array([[-127, 5, 1, -2]], np.int8)
    sh = np.array([[0.5], [0.25]])
    np.testing.assert_array_equal(oracle.dequant_int8_group(qh, sh, 2), [[-63.5, 2.5, 0.25, -0.5]])
    # one scale repeated over every group is the per-column format
    s_col = rng.random(16) + 0.1
    assert np.array_equal(oracle.dequant_int8_group(q, np.tile(s_col, (3, 1)), 128), oracle.dequant_int8(q, s_col))


# ----------------------------------------------------------------------------
# 2:4 structured sparsity ("Add GPTQ Marlin 2:4 sparse structured support")
# ----------------------------------------------------------------------------
def test_decompress_24_worked_example():
    # one row, K = 8: group 0 keeps channels 0 and 2, group 1 keeps 5 and 7
    values = np.array([[3, 12, 0, 15]], np.uint8)
    positions = np.array([[[0, 2], [1, 3]]])
    got = oracle.decompress_24(values, positions)
    np.testing.assert_array_equal(got, [[3, 8, 12, 8, 8, 0, 8, 15]])


def _compress_24_loops(q):
    """Scalar compressor: per group of 4, the channels whose code is not 8, padded
    with the lowest remaining channels; None if a group has more than two."""
    N, K = q.shape
    values = np.zeros((N, K // 2), np.uint8)
    positions = np.zeros((N, K // 4, 2), np.int64)
    for n in range(N):
        for j in range(K // 4):
            nz = [i for i in range(4) if q[n, 4 * j + i] != 8]
            if len(nz) > 2:
                return None
            for i in range(4):
                if len(nz) < 2 and i not in nz:
                    nz.append(i)
            nz = sorted(nz[:2])
            positions[n, j] = nz
            values[n, 2 * j] = q[n, 4 * j + nz[0]]
            values[n, 2 * j + 1] = q[n, 4 * j + nz[1]]
    return values, positions


def test_decompress_24_inverts_scalar_compressor():
    rng = np.random.default_rng(5)
    N, K = 7, 64
    q = np.full((N, K), 8, np.uint8)
    for n in range(N):
        for j in range(K // 4):
            keep = rng.choice(4, size=rng.integers(0, 3), replace=False)
            q[n, 4 * j + keep] = rng.integers(0, 16, size=keep.size)
    values, positions = _compress_24_loops(q)
    np.testing.assert_array_equal(oracle.decompress_24(values, positions), q)
    # a swapped position pair puts the values at the wrong channels
    bad = positions.copy()
    bad[0, 0] = bad[0, 0][::-1]
    if values[0, 0] != values[0, 1]:
        assert not np.array_equal(oracle.decompress_24(values, bad), q)


def test_prune_24_keeps_two_largest_per_group():
    rng = np.random.default_rng(6)
    w = rng.standard_normal((5, 32)).astype(np.float32)
    w[0, 0:4] = [1.0, -1.0, 1.0, 0.5]          # ties: the lower channels win
    p = prune_24(w)
    for n in range(w.shape[0]):
        for j in range(w.shape[1] // 4):
            g = [abs(float(v)) for v in w[n, 4 * j:4 * j + 4]]
            order = sorted(range(4), key=lambda i: (-g[i], i))[:2]
            for i in range(4):
                want = w[n, 4 * j + i] if i in order else 0.0
                assert p[n, 4 * j + i] == want
    np.testing.assert_array_equal(p[0, 0:4], [1.0, -1.0, 0.0, 0.0])
    np.testing.assert_array_equal(prune_24(p), p)


@pytest.mark.parametrize("gs", [16, -1])
def test_quantize_int4_24_structure_and_round_trip(gs):
    rng = np.random.default_rng(7)
    w = (0.02 * rng.standard_normal((12, 64))).astype(np.float32)
    q, s = quantize_int4_24(w, gs, "f16")
    nz = (q.reshape(12, 16, 4) != 8).sum(axis=2)
    assert nz.max() <= 2
    p = prune_24(w)
    assert np.all(q[p == 0] == 8)
    deq = oracle.dequant_int4(q, s, None, gs)
    g = np.arange(64) // (64 if gs < 0 else gs)
    assert np.all(np.abs(deq - p) <= s[g, :].T / 2 + 1e-12)


# ----------------------------------------------------------------------------
# 2:4-sparse int8 and the dense linear layer
# ("Add GPTQ Marlin 2:4 sparse structured support": 4 or 8 bits, group 128 or
# channel-wise, dense or 2:4 sparse, a dense linear layer)
# ----------------------------------------------------------------------------
def test_decompress_24_int8_worked_example_and_inverse():
    # signed codes, zero code 0: group 0 keeps channels 1 and 3, group 1 keeps 4 and 5
    values = np.array([[-7, 127, -127, 3]], np.int8)
    positions = np.array([[[1, 3], [0, 1]]])
    got = oracle.decompress_24(values, positions, zero_code=0)
    assert got.dtype == np.int8
    np.testing.assert_array_equal(got, [[0, -7, 0, 127, -127, 3, 0, 0]])
    rng = np.random.default_rng(9)
    q = np.zeros((5, 32), np.int8)
    for n in range(5):
        for j in range(8):
            keep = rng.choice(4, size=rng.integers(0, 3), replace=False)
            q[n, 4 * j + keep] = rng.integers(-127, 128, size=keep.size)
    vals = np.zeros((5, 16), np.int8)
    pos = np.zeros((5, 8, 2), np.int64)
    for n in range(5):
        for j in range(8):
            nz = [i for i in range(4) if q[n, 4 * j + i] != 0]
            nz += [i for i in range(4) if i not in nz][:2 - len(nz)]
            nz = sorted(nz)
            pos[n, j] = nz
            vals[n, 2 * j:2 * j + 2] = q[n, 4 * j + nz[0]], q[n, 4 * j + nz[1]]
    np.testing.assert_array_equal(oracle.decompress_24(vals, pos, zero_code=0), q)


@pytest.mark.parametrize("gs", [-1, 128])
def test_quantize_int8_24_structure_and_round_trip(gs):
    rng = np.random.default_rng(10)
    w = (rng.standard_normal((12, 256)) * 0.02).astype(np.float32)
    q, s = quantize_int8_24(w, gs, "bf16")
    assert q.dtype == np.int8 and np.abs(q.astype(np.int32)).max() <= 127
    assert np.all((q.reshape(12, 64, 4) != 0).sum(axis=2) <= 2)
    wp = prune_24(w)
    if gs < 0:
        assert s.shape == (12,)
        wd = oracle.dequant_int8(q, s)
        tol = np.repeat(s[:, None], 256, axis=1)
    else:
        assert s.shape == (2, 12)
        wd = oracle.dequant_int8_group(q, s, gs)
        tol = np.repeat(s.T, gs, axis=1)
    assert np.all(np.abs(wd - wp) <= tol * (0.5 + 1e-6))
    assert np.all(wd[wp == 0] == 0)


def test_linear_forward_closed_form_and_brute_force():
    # W = diag(d) . P (a scaled permutation): out[m, n] = d[n] * x[m, pi[n]]
    rng = np.random.default_rng(11)
    K = 16
    pi = rng.permutation(K)
    d = rng.integers(-7, 8, size=K).astype(np.float64)
    W = np.zeros((K, K))
    W[np.arange(K), pi] = d
    x = rng.standard_normal((3, K))
    np.testing.assert_allclose(oracle.linear_forward(x, W), d[None, :] * x[:, pi], rtol=0, atol=1e-14)
    # scalar loops on a quantized layer of every format, dequantized inside the dot product
    for qt, gs, ao in [("int4", 32, True), ("int4zp", 32, False), ("int4s24", -1, False), ("int8", -1, False),
                       ("int8g", 32, False), ("int8s24", 32, False), ("int8s24", -1, False)]:
        lin = make_linear(8, 64, qt, gs, "bf16", act_order=ao, seed=3)
        xs = make_linear_inputs(64, 2, "bf16", seed=4)
        got = oracle.linear_forward(xs, oracle.dequant_linear(lin))
        want = np.zeros((2, 8))
        for m in range(2):
            for n in range(8):
                acc = 0.0
                for k in range(64):
                    if qt.startswith("int4"):
                        g = int(lin.g_idx[k]) if lin.g_idx is not None else (0 if gs < 0 else k // gs)
                        zero = 8 if lin.z is None else int(lin.z[g, n])
                        wv = (int(lin.q[n, k]) - zero) * float(lin.s[g, n])
                    elif lin.s.ndim == 1:
                        wv = int(lin.q[n, k]) * float(lin.s[n])
                    else:
                        wv = int(lin.q[n, k]) * float(lin.s[k // gs, n])
                    acc += float(xs[m, k]) * wv
                want[m, n] = acc
        np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12, err_msg=qt)


def test_int8_24_expert_layer_brute_force():
    wl = _wl(E=3, k=2, H=32, I=48, qt="int8s24", group_size=-1)
    layer = make_layer(wl, seed=19)
    assert np.all((layer.q13.reshape(3, 96, 8, 4) != 0).sum(axis=3) <= 2)
    inp = make_inputs(wl, 3, seed=19)
    got = oracle.moe_forward(layer, inp.x, inp.topk_ids, inp.topk_weights)
    want = _brute_force(layer, inp.x, inp.topk_ids, inp.topk_weights)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)
