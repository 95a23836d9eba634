"""Host-side checks of libqmoe (no GPU): the library loads, exports every
function include/qmoe.h declares, packs weights in the documented layout with
a bit-exact round trip, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import numpy as np
import pytest

import weight_only_quantized_moe_gb300 as q
from weight_only_quantized_moe_gb300 import _native as N
from synth import Workload, make_layer, to_u16_bits


@pytest.fixture(scope="session", autouse=True)
def built_library():
    from weight_only_quantized_moe_gb300 import build
    build.build()
    return q.lib()


def _declared_functions():
    text = open(N.HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qmoe_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = _declared_functions()
    assert len(names) >= 15
    dll = ctypes.CDLL(N.LIB_PATH)
    missing = [n for n in names if not hasattr(dll, n)]
    assert not missing, missing
    assert q.lib().qmoe_abi_version() == 2
    for s in range(0, 8):
        assert q.status_string(s)


def _wl(qt, act_order=False, E=3, H=256, I=384):
    return Workload("t", E, 2, H, I, qt, 128 if qt == "int4" else -1, "bf16" if qt == "int8" else "f16",
                    act_order, 0.0, (1,))


@pytest.mark.parametrize("act_order", [False, True])
@pytest.mark.parametrize("act", ["f16", "bf16"])
def test_pack_int4_round_trip(act_order, act):
    wl = _wl("int4", act_order)
    wl = Workload(wl.name, wl.E, wl.k, wl.H, wl.I, "int4", 128, act, act_order, 0.0, (1,))
    L = make_layer(wl, seed=2)
    s13b, s2b = to_u16_bits(L.s13, act), to_u16_bits(L.s2, act)
    pk = q.qmoe_pack_int4(wl.E, wl.H, wl.I, act, L.q13, s13b, L.g13, L.q2, s2b, L.g2)
    assert pk["w13"].nbytes == wl.E * (2 * wl.I // 128) * (wl.H // 128) * 8448
    q13, s13, q2, s2 = q.qmoe_unpack_int4(wl.E, wl.H, wl.I, pk["w13"], pk["w2"], L.g13, L.g2)
    assert np.array_equal(q13, L.q13) and np.array_equal(q2, L.q2)
    assert np.array_equal(s13, s13b) and np.array_equal(s2, s2b)
    if act_order:
        # perm13 lists each expert's hidden channels by group, ascending inside a group
        for e in range(wl.E):
            p = pk["perm13"][e]
            assert sorted(p.tolist()) == list(range(wl.H))
            g = L.g13[e][p]
            assert np.all(np.diff(g) >= 0)
            assert all(np.all(np.diff(p[g == gg]) > 0) for gg in range(wl.H // 128))


def test_pack_int4_layout_matches_documented_nibble_order():
    # one expert, gate row 0 and up row 0 carry distinct codes along K
    E, H, I = 1, 128, 128
    q13 = np.full((E, 2 * I, H), 8, np.uint8)
    q13[0, 0, :] = np.arange(H) % 16          # gate channel 0 -> packed row 0
    q13[0, I, :] = (np.arange(H) * 7) % 16    # up channel 0 -> packed row 1
    s13 = np.full((E, 1, 2 * I), 0x3C00, np.uint16)
    s13[0, 0, I] = 0x4000
    q2 = np.full((E, H, I), 8, np.uint8)
    s2 = np.full((E, 1, H), 0x3C00, np.uint16)
    pk = q.qmoe_pack_int4(E, H, I, "f16", q13, s13, None, q2, s2, None)
    blk = pk["w13"][:8448]                   # tile 0, K stage 0
    for r, codes in ((0, q13[0, 0]), (1, q13[0, I])):
        for c in range(4):
            for j in range(4):
                word = int.from_bytes(bytes(blk[(c * 128 + r) * 16 + 4 * j:(c * 128 + r) * 16 + 4 * j + 4]), "little")
                for i in range(4):
                    k0 = 32 * c + 8 * j + 2 * i
                    assert (word >> (4 * i)) & 15 == codes[k0]
                    assert (word >> (4 * (i + 4))) & 15 == codes[k0 + 1]
    assert int.from_bytes(bytes(blk[8192:8194]), "little") == 0x3C00
    assert int.from_bytes(bytes(blk[8194:8196]), "little") == 0x4000


def test_pack_int8_round_trip():
    wl = _wl("int8")
    L = make_layer(wl, seed=4)
    pk = q.qmoe_pack_int8(wl.E, wl.H, wl.I, L.q13, L.s13, L.q2, L.s2)
    q13, s13, q2, s2 = q.qmoe_unpack_int8(wl.E, wl.H, wl.I, pk["w13"], pk["s13"], pk["w2"], pk["s2"])
    assert np.array_equal(q13, L.q13) and np.array_equal(q2, L.q2)
    assert np.array_equal(s13, L.s13) and np.array_equal(s2, L.s2)
    # packed row order interleaves gate and up channels
    assert np.array_equal(pk["s13"][0, 0::2], L.s13[0, :wl.I])
    assert np.array_equal(pk["s13"][0, 1::2], L.s13[0, wl.I:])


def test_pack_rejects_bad_codes_and_groups():
    E, H, I = 1, 128, 128
    q13 = np.full((E, 2 * I, H), 8, np.uint8)
    s = np.full((E, 1, 2 * I), 0x3C00, np.uint16)
    q2 = np.full((E, H, I), 8, np.uint8)
    s2 = np.full((E, 1, H), 0x3C00, np.uint16)
    bad = q13.copy()
    bad[0, 3, 5] = 16
    with pytest.raises(q.QmoeError) as ei:
        q.qmoe_pack_int4(E, H, I, "f16", bad, s, None, q2, s2, None)
    assert ei.value.status == q.QMOE_ERR_INVALID_ARG
    g = np.zeros((E, H), np.int32)
    g[0, :64] = 0
    g[0, 64:] = 1  # group 1 does not exist for H = 128
    with pytest.raises(q.QmoeError) as ei:
        q.qmoe_pack_int4(E, H, I, "f16", q13, s, g, q2, s2, None)
    assert ei.value.status == q.QMOE_ERR_UNSUPPORTED
    q8 = np.zeros((E, 2 * I, H), np.int8)
    q8[0, 0, 0] = -128
    with pytest.raises(q.QmoeError) as ei:
        q.qmoe_pack_int8(E, H, I, q8, np.ones((E, 2 * I), np.float32), np.zeros((E, H, I), np.int8),
                         np.ones((E, H), np.float32))
    assert ei.value.status == q.QMOE_ERR_INVALID_ARG


def _layer_struct(**kw):
    base = dict(E=8, H=256, I=512, group_size=128, qt=N.QMOE_INT4_GROUP, act_dtype=N.QMOE_F16,
                scale_dtype=N.QMOE_F16, w13=None, w2=None, s13=None, s2=None, perm13=None)
    base.update(kw)
    return N.QmoeLayer(**base)


def test_workspace_size_and_validation_are_host_only():
    L = q.lib()
    ok = _layer_struct()
    n = L.qmoe_workspace_size(ctypes.byref(ok), 16, 2)
    assert n > 0 and n % 256 == 0
    assert L.qmoe_workspace_size(ctypes.byref(ok), 4096, 2) > n
    assert L.qmoe_workspace_size_host(ctypes.byref(ok), 16, 2) > n
    for bad in (_layer_struct(H=200), _layer_struct(I=100), _layer_struct(E=0), _layer_struct(E=2000),
                _layer_struct(group_size=64), _layer_struct(scale_dtype=N.QMOE_BF16),
                _layer_struct(qt=N.QMOE_INT8_PER_COL, group_size=-1, scale_dtype=N.QMOE_F16),
                _layer_struct(act_dtype=N.QMOE_F32, scale_dtype=N.QMOE_F32)):
        assert L.qmoe_workspace_size(ctypes.byref(bad), 16, 2) == 0
    assert L.qmoe_workspace_size(ctypes.byref(ok), 16, 9) == 0     # top_k > E
    assert L.qmoe_workspace_size(ctypes.byref(ok), -1, 2) == 0
    # forward rejects before any device access
    st = L.qmoe_forward(ctypes.byref(_layer_struct(H=200)), None, 4, None, None, 2, None, None, 0, None)
    assert st == q.QMOE_ERR_UNSUPPORTED
    st = L.qmoe_forward(ctypes.byref(ok), None, 4, None, None, 2, None, None, 0, None)
    assert st == q.QMOE_ERR_WORKSPACE
    # the no-allocation forward reports an invalid layer or size exactly as qmoe_forward
    # does, before any device access, also at M == 0
    for bad, M, k in ((_layer_struct(H=200), 0, 2), (_layer_struct(E=0), 0, 2), (_layer_struct(group_size=64), 0, 2),
                      (_layer_struct(qt=99), 0, 2), (ok, 0, 9), (_layer_struct(H=200), 4, 2), (ok, -1, 2)):
        want = L.qmoe_forward(ctypes.byref(bad), None, M, None, None, k, None, None, 0, None)
        got = L.qmoe_forward_noalloc(ctypes.byref(bad), None, M, None, None, k, None, None)
        assert want != q.QMOE_OK and got == want, (M, k, want, got)
    assert L.qmoe_forward_noalloc(None, None, 0, None, None, 2, None, None) == q.QMOE_ERR_INVALID_ARG
    # moe_align argument checks
    assert L.qmoe_moe_align(None, 4, 2, 8, 16, None, None, None, 1000, None) == q.QMOE_ERR_INVALID_ARG
    assert L.qmoe_moe_align(None, 4, 2, 8, 0, None, None, None, 1000, None) == q.QMOE_ERR_INVALID_ARG
    assert L.qmoe_moe_align(None, 4, 2, 8, 16, None, None, None, 10, None) == q.QMOE_ERR_INVALID_ARG


# ----------------------------------------------------------------------------
# other weight formats: zero points, channel-wise int4, grouped int8
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("act_order,gs", [(False, 128), (True, 128), (False, -1)])
@pytest.mark.parametrize("act", ["f16", "bf16"])
def test_pack_int4_zero_points_round_trip(act_order, gs, act):
    wl = Workload("zp", 4, 2, 256, 384, "int4zp", gs, act, act_order, 0.0, (1,))
    L = make_layer(wl, seed=6)
    s13b, s2b = to_u16_bits(L.s13, act), to_u16_bits(L.s2, act)
    pk = q.qmoe_pack_int4(wl.E, wl.H, wl.I, act, L.q13, s13b, L.g13, L.q2, s2b, L.g2, gs, L.z13, L.z2)
    assert pk["w13"].nbytes == wl.E * (2 * wl.I // 128) * (wl.H // 128) * 8576
    q13, s13, q2, s2, z13, z2 = q.qmoe_unpack_int4(wl.E, wl.H, wl.I, pk["w13"], pk["w2"], L.g13, L.g2, gs, zp=True)
    assert np.array_equal(q13, L.q13) and np.array_equal(q2, L.q2)
    assert np.array_equal(s13, s13b) and np.array_equal(s2, s2b)
    assert np.array_equal(z13, L.z13) and np.array_equal(z2, L.z2)


def test_pack_int4_channel_wise_round_trip_and_block_scales():
    wl = Workload("cw", 2, 2, 256, 256, "int4", -1, "f16", False, 0.0, (1,))
    L = make_layer(wl, seed=7)
    assert L.s13.shape == (2, 1, 512)
    s13b, s2b = to_u16_bits(L.s13, "f16"), to_u16_bits(L.s2, "f16")
    pk = q.qmoe_pack_int4(wl.E, wl.H, wl.I, "f16", L.q13, s13b, None, L.q2, s2b, None, -1)
    q13, s13, q2, s2 = q.qmoe_unpack_int4(wl.E, wl.H, wl.I, pk["w13"], pk["w2"], None, None, -1)
    assert np.array_equal(q13, L.q13) and np.array_equal(s13, s13b) and np.array_equal(s2, s2b)
    # every K block of a W2 tile carries the row's one scale (bytes 8192.. of each 8448-byte block)
    blk = pk["w2"][: (wl.I // 128) * 8448].reshape(wl.I // 128, 8448)
    sc = blk[:, 8192:8448].view(np.uint16)
    assert np.array_equal(sc[0], sc[1]) and np.array_equal(sc[0], s2b[0, 0, :128])
    # channel-wise scales cannot carry an act-order g_idx
    with pytest.raises(q.QmoeError) as ei:
        q.qmoe_pack_int4(wl.E, wl.H, wl.I, "f16", L.q13, s13b, np.zeros((2, 256), np.int32), L.q2, s2b, None, -1)
    assert ei.value.status == q.QMOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("act", ["f16", "bf16"])
def test_pack_int8_group_round_trip(act):
    wl = Workload("i8g", 3, 2, 256, 384, "int8g", 128, act, False, 0.0, (1,))
    L = make_layer(wl, seed=8)
    s13b, s2b = to_u16_bits(L.s13, act), to_u16_bits(L.s2, act)
    pk = q.qmoe_pack_int8_group(wl.E, wl.H, wl.I, act, L.q13, s13b, L.q2, s2b)
    assert pk["w13"].nbytes == wl.E * (2 * wl.I // 128) * (wl.H // 128) * 16640
    q13, s13, q2, s2 = q.qmoe_unpack_int8_group(wl.E, wl.H, wl.I, pk["w13"], pk["w2"])
    assert np.array_equal(q13, L.q13) and np.array_equal(q2, L.q2)
    assert np.array_equal(s13, s13b) and np.array_equal(s2, s2b)


def test_pack_rejects_bad_zero_points():
    wl = Workload("zp", 1, 2, 128, 128, "int4zp", 128, "f16", False, 0.0, (1,))
    L = make_layer(wl, seed=9)
    s13b, s2b = to_u16_bits(L.s13, "f16"), to_u16_bits(L.s2, "f16")
    z13 = L.z13.copy()
    z13[0, 0, 3] = 16
    with pytest.raises(q.QmoeError) as ei:
        q.qmoe_pack_int4(1, 128, 128, "f16", L.q13, s13b, None, L.q2, s2b, None, 128, z13, L.z2)
    assert ei.value.status == q.QMOE_ERR_INVALID_ARG
    assert q.packed_bytes("int4zp", 1, 256, 128) == 2 * 8576
    assert q.packed_bytes("int8g", 1, 256, 128) == 2 * 16640
    assert q.packed_bytes("int4", 1, 256, 128, -1) == 2 * 8448
    assert q.packed_bytes("int8g", 1, 256, 128, -1) == 0


def test_options_layout_and_issuer_validation():
    """qmoe_options is 16 int32 fields (11 knobs and 5 reserved); the knobs are checked on the host."""
    assert ctypes.sizeof(N.QmoeOptions) == 64
    L = q.lib()
    ok = _layer_struct()

    def size(M, **kw):
        return L.qmoe_workspace_size_ex(ctypes.byref(ok), M, 2, ctypes.byref(q.make_options(**kw)))

    assert size(16) == L.qmoe_workspace_size(ctypes.byref(ok), 16, 2)
    for n in (1, 2, 3):
        assert size(16, issuers=n) > 0          # 16-row token tile: any issuer count fits
    assert size(4096, issuers=2) > 0           # 128-row tile, two issuers: 256 accumulator columns
    assert size(4096, issuers=3) == 0          # 384 accumulator columns leave no room for A slots
    assert size(16, issuers=4) == 0
    assert size(16, issuers=-1) == 0
    for bad in (dict(dq_sets=3), dict(weight_l2=3), dict(token_ring=4), dict(dq_sets=-1), dict(topk_reduce=3),
                dict(topk_reduce=-1)):
        assert size(16, **bad) == 0, bad
    for good in (dict(dq_sets=2), dict(dq_sets=4), dict(weight_l2=1), dict(weight_l2=2), dict(token_ring=1),
                 dict(topk_reduce=1), dict(topk_reduce=2)):
        assert size(16, **good) > 0, good
    # the in-GEMM reduction adds its arrival counters (M x H/128 x 4 int32) to the workspace
    assert size(16, topk_reduce=1) > size(16, topk_reduce=2)
    assert size(16) == size(16, topk_reduce=2)


def test_cta_pair_option():
    """CTA pairs: symmetric int4 and per-column int8 only, not with the in-GEMM top-k
    reduction or the per-group int4 epilogue, not for the dense linear layer; the plan
    reports them and each CTA's token-tile slots hold half the rows, so 128-row tiles
    get a deeper token ring."""
    L = q.lib()
    ok = _layer_struct()

    def size(M, layer=ok, **kw):
        return L.qmoe_workspace_size_ex(ctypes.byref(layer), M, 2, ctypes.byref(q.make_options(**kw)))

    for good in (dict(cta_pair=1), dict(cta_pair=2), dict(cta_pair=1, token_tile=128), dict(cta_pair=1, topk_reduce=2)):
        assert size(16, **good) > 0, good
    for bad in (dict(cta_pair=3), dict(cta_pair=-1), dict(cta_pair=1, topk_reduce=1),
                dict(cta_pair=1, token_tile=16, int4_group_epilogue=1)):
        assert size(16, **bad) == 0, bad
    for qt, gs in ((N.QMOE_INT4_GROUP_ZP, 128), (N.QMOE_INT8_GROUP, 128), (N.QMOE_INT4_GROUP_24, 128)):
        assert size(16, _layer_struct(qt=qt, group_size=gs), cta_pair=1) == 0, qt
    i8 = _layer_struct(qt=N.QMOE_INT8_PER_COL, group_size=-1, scale_dtype=N.QMOE_F32)
    assert size(16, i8, cta_pair=1) > 0
    # automatic: pairs where a single CTA's rings are short (128-row int4 tiles: a token ring of one
    # A-ring depth; 64-row int8 tiles), single CTAs where they are deep (decode, 64-row int4 tiles)
    single, pair = _plan(MIXTRAL, 2048, cta_pair=2), _plan(MIXTRAL, 2048, cta_pair=1)
    assert single["b_stages"] == single["ab_stages"] and pair["b_stages"] == 2 * single["b_stages"]
    assert _plan(MIXTRAL, 2048)["cta_pair"] == 1 and _plan(MIXTRAL, 2048)["b_stages"] == pair["b_stages"]
    assert _plan(MIXTRAL, 16)["cta_pair"] == 0 and _plan(MIXTRAL, 128)["cta_pair"] == 0
    I8 = dict(E=8, H=4096, I=14336, group_size=-1, qt=N.QMOE_INT8_PER_COL, scale_dtype=N.QMOE_F32)
    assert [_plan(I8, M)["cta_pair"] for M in (16, 128, 512)] == [0, 1, 1]
    assert _plan(MIXTRAL, 2048, token_ring=1)["cta_pair"] == 0      # rings set by hand: no automatic pair
    # the down GEMM follows, except where its K spans fewer than 32 stages (I = 1536: 12)
    assert _plan(MIXTRAL, 2048)["cta_pair_down"] == 1 and _plan(MIXTRAL, 16)["cta_pair_down"] == 0
    DS = dict(E=160, H=5120, I=1536, group_size=-1, qt=N.QMOE_INT8_PER_COL, scale_dtype=N.QMOE_F32)
    p1024 = _plan(DS, 1024, k=6)
    assert p1024["cta_pair"] == 1 and p1024["cta_pair_down"] == 0
    assert _plan(DS, 1024, k=6, cta_pair=1)["cta_pair_down"] == 1        # the option pairs both
    lin = N.QmoeLinear(4096, 14336, 128, N.QMOE_INT4_GROUP, N.QMOE_F16, N.QMOE_F16, None, None, None)
    assert L.qmoe_linear_workspace_size(ctypes.byref(lin), 16, ctypes.byref(q.make_options(cta_pair=1))) == 0
    assert L.qmoe_linear_workspace_size(ctypes.byref(lin), 16, ctypes.byref(q.make_options(cta_pair=2))) > 0


def _sparse_position(area, r, G):
    """Position nibble (i0 | i1 << 2) of group G (0..31, 4 input channels each) of row r in a
    2048-byte position area, in the order the structured-sparse MMA reads it: MMA k = G // 8 covers
    groups 8k .. 8k+7 as sub-blocks s = (G // 4) % 2; lane L = 16b + 8s + i holds sub-block s of row
    16b + i in bits 0-15 and of row 16b + 8 + i in bits 16-31; its word for MMA k is at byte
    (k // 2) * 1024 + 8L + 4 (k % 2)."""
    k, s, t = G // 8, (G // 4) % 2, G % 4
    b, hi, i = r // 16, (r // 8) % 2, r % 8
    L = 16 * b + 8 * s + i
    off = (k // 2) * 1024 + 8 * L + 4 * (k % 2)
    word = int.from_bytes(bytes(area[off:off + 4]), "little")
    return (word >> (16 * hi + 4 * t)) & 15


@pytest.mark.parametrize("act,gs", [("f16", 128), ("bf16", 128), ("f16", -1)])
def test_pack_int4_24_round_trip_and_layout(act, gs):
    import oracle
    wl = Workload("s24", 2, 2, 256, 384, "int4s24", gs, act, False, 0.0, (1,))
    L = make_layer(wl, seed=10)
    s13b, s2b = to_u16_bits(L.s13, act), to_u16_bits(L.s2, act)
    pk = q.qmoe_pack_int4_24(wl.E, wl.H, wl.I, act, L.q13, s13b, L.q2, s2b, gs)
    assert pk["w13"].nbytes == wl.E * (2 * wl.I // 128) * (wl.H // 128) * 6400
    q13, s13, q2, s2 = q.qmoe_unpack_int4_24(wl.E, wl.H, wl.I, pk["w13"], pk["w2"], gs)
    assert np.array_equal(q13, L.q13) and np.array_equal(q2, L.q2)
    assert np.array_equal(s13, s13b) and np.array_equal(s2, s2b)
    # the packed block read back through the oracle's definition of the format:
    # W2 of expert 0, tile 0, K block 0, half h, row r holds channels 64h .. 64h+63 of row r
    blk = pk["w2"][:6400]
    for r in (0, 77, 127):
        for h in (0, 1):
            codes = blk[(h * 128 + r) * 16:(h * 128 + r) * 16 + 16]
            vals = np.zeros((1, 32), np.uint8)
            positions = np.zeros((1, 16, 2), np.int64)
            for g in range(16):
                j, i = divmod(g, 4)
                word = int.from_bytes(bytes(codes[4 * j:4 * j + 4]), "little")
                vals[0, 2 * g] = (word >> (4 * i)) & 15
                vals[0, 2 * g + 1] = (word >> (4 * (i + 4))) & 15
                m = _sparse_position(blk[4096:6144], r, 16 * h + g)
                positions[0, g] = (m & 3, m >> 2)
                assert (m & 3) < (m >> 2)
            dense = oracle.decompress_24(vals, positions)
            assert np.array_equal(dense[0], L.q2[0, r, 64 * h:64 * h + 64])
        assert int.from_bytes(bytes(blk[6144 + 2 * r:6146 + 2 * r]), "little") == s2b[0, 0, r]


def test_pack_int4_24_rejects_three_of_four():
    wl = Workload("s24", 1, 2, 128, 128, "int4s24", 128, "f16", False, 0.0, (1,))
    L = make_layer(wl, seed=11)
    s13b, s2b = to_u16_bits(L.s13, "f16"), to_u16_bits(L.s2, "f16")
    q2 = L.q2.copy()
    q2[0, 5, 8:12] = [1, 2, 3, 8]
    with pytest.raises(q.QmoeError) as ei:
        q.qmoe_pack_int4_24(1, 128, 128, "f16", L.q13, s13b, q2, s2b)
    assert ei.value.status == q.QMOE_ERR_INVALID_ARG
    assert q.packed_bytes("int4s24", 1, 256, 128) == 2 * 6400


def test_pack_int4_24_sparse_corner_groups():
    """Groups with 0 or 1 codes other than 8 (padded with the lowest free channels)
    and every kept-position pair round-trip exactly; channel-wise scales repeat."""
    wl = Workload("s24c", 1, 2, 256, 128, "int4s24", -1, "f16", False, 0.0, (1,))
    L = make_layer(wl, seed=12)
    s13b, s2b = to_u16_bits(L.s13, "f16"), to_u16_bits(L.s2, "f16")
    q2 = np.full_like(L.q2, 8)
    pairs = [(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)]
    for r in range(q2.shape[1]):
        for g in range(q2.shape[2] // 4):
            kind = (r + g) % 9
            base = 4 * g
            if kind < 6:
                i0, i1 = pairs[kind]
                q2[0, r, base + i0] = (r + g) % 16 if (r + g) % 16 != 8 else 1
                q2[0, r, base + i1] = (3 * r + g) % 16 if (3 * r + g) % 16 != 8 else 2
            elif kind < 8:
                q2[0, r, base + (r + kind) % 4] = 15   # one code only
            # kind == 8: the whole group is zero
    pk = q.qmoe_pack_int4_24(1, 256, 128, "f16", L.q13, s13b, q2, s2b, -1)
    q13, s13, q2b, s2 = q.qmoe_unpack_int4_24(1, 256, 128, pk["w13"], pk["w2"], -1)
    assert np.array_equal(q2b, q2) and np.array_equal(q13, L.q13)
    assert np.array_equal(s2, s2b) and np.array_equal(s13, s13b)
    # channel-wise: both 128-K blocks of a W13 tile (K = H = 256) carry the rows' one scale
    blk = pk["w13"].reshape(-1, 6400)
    assert np.array_equal(blk[0, 6144:6400], blk[1, 6144:6400])
    assert not np.array_equal(blk[0, 6144:6400], blk[2, 6144:6400])


def test_packed_bytes_per_format():
    tiles = 3 * (256 // 128) * (384 // 128)
    for qt, gs, per in [("int4", 128, 8448), ("int4", -1, 8448), ("int4zp", 128, 8576), ("int4s24", 128, 6400),
                        ("int4s24", -1, 6400), ("int8", -1, 16384), ("int8g", 128, 16640)]:
        assert q.packed_bytes(qt, 3, 256, 384, gs) == tiles * per
    for qt, gs in [("int4", 64), ("int4s24", 256), ("int8", 128), ("int8g", -1)]:
        assert q.packed_bytes(qt, 3, 256, 384, gs) == 0
    assert q.packed_bytes("int4s24", 3, 200, 384, 128) == 0


def _plan(layer_kw, M, k=2, sms=152, **opts):
    return q.qmoe_describe_plan(_layer_struct(**layer_kw), M, k, q.make_options(**opts) if opts else None, sms)


MIXTRAL = dict(E=8, H=4096, I=14336, group_size=128, qt=N.QMOE_INT4_GROUP)


@pytest.mark.parametrize("M,T,ni,s2", [(1, 16, 2, 2), (4, 16, 2, 3), (16, 16, 2, 4), (32, 16, 2, 4), (64, 32, 2, 4),
                                       (128, 64, 2, 4), (256, 128, 1, 1), (2048, 128, 1, 1)])
def test_plan_token_tile_issuers_and_split(M, T, ni, s2):
    """Token tile: the power of two >= 1.5 x mean pairs per expert (16..128); issuers 2 up to 64-row
    tiles, else 1; down-GEMM split as fitted on GB300 for the Mixtral-8x7B shape."""
    p = _plan(MIXTRAL, M)
    assert (p["token_tile"], p["issuers"], p["split2"]) == (T, ni, s2)
    assert p["split1"] == 1 and p["stage_bytes"] == 8448
    assert p["workspace_bytes"] == L_ws(MIXTRAL, M)


def L_ws(kw, M):
    return q.lib().qmoe_workspace_size(ctypes.byref(_layer_struct(**kw)), M, 2)


def test_plan_rings_and_tmem_constraints():
    """Every plan keeps the ring rules the kernel relies on: even weight ring, A ring a multiple of
    lcm(2, issuers), TMEM columns (accumulators + 64-column A slots) within 512, shared memory within
    227 KB."""
    for qt, gs, per in [(N.QMOE_INT4_GROUP, 128, 8448), (N.QMOE_INT4_GROUP_24, 128, 6400),
                        (N.QMOE_INT8_PER_COL, -1, 16384), (N.QMOE_INT8_GROUP, 128, 16640)]:
        sdt = N.QMOE_F32 if qt == N.QMOE_INT8_PER_COL else N.QMOE_F16
        for M in (1, 16, 64, 128, 512, 4096):
            for ni in (0, 1, 2, 3):
                try:
                    p = _plan(dict(E=8, H=4096, I=14336, group_size=gs, qt=qt, scale_dtype=sdt), M, issuers=ni)
                except q.QmoeError:
                    assert ni != 0          # the automatic choice always has a plan
                    continue
                T, NI = p["token_tile"], p["issuers"]
                mult = 6 if NI == 3 else 2
                assert p["w_stages"] % 2 == 0 and p["w_stages"] >= 2
                assert p["ab_stages"] % mult == 0 and p["ab_stages"] >= mult
                assert NI * p["acc_bufs"] * T + 64 * p["ab_stages"] <= 512
                wslot = (per + 1023) // 1024 * 1024
                assert p["b_stages"] % p["ab_stages"] == 0 and p["b_stages"] <= 3 * p["ab_stages"]
                assert 1024 + p["w_stages"] * wslot + p["b_stages"] * T * (128 if p["cta_pair"] else 256) + 1024 <= 232448
                # barriers below the selector table at the end of the 1 KB barrier area
                assert (2 * p["w_stages"] + p["ab_stages"] + p["b_stages"] + 7) * 8 + 8 <= 1024 - 128
                assert p["stage_bytes"] == per


def test_plan_overrides_and_other_workloads():
    p = _plan(MIXTRAL, 16, split1=3, split2=5, token_tile=48, issuers=2)
    assert (p["split1"], p["split2"], p["token_tile"], p["issuers"]) == (3, 5, 48, 2)
    # token-tile ring twice the A ring at decode sizes, equal at 128-row tiles on single CTAs (shared
    # memory), twice again on CTA pairs (half of each tile per CTA)
    p16 = _plan(MIXTRAL, 16)
    assert p16["b_stages"] == 2 * p16["ab_stages"] and p16["w_stages"] >= 8
    p2k = _plan(MIXTRAL, 2048, cta_pair=2)
    assert p2k["b_stages"] == p2k["ab_stages"]
    for m in (1, 2, 3):
        pm = _plan(MIXTRAL, 16, token_ring=m)
        assert pm["b_stages"] == m * pm["ab_stages"]
    with pytest.raises(q.QmoeError):
        _plan(MIXTRAL, 2048, token_ring=3)       # 12 x 32 KB token tiles do not fit
    with pytest.raises(q.QmoeError):
        _plan(MIXTRAL, 16, token_ring=4)
    ds = dict(E=160, H=5120, I=1536, group_size=-1, qt=N.QMOE_INT8_PER_COL, scale_dtype=N.QMOE_F32)
    assert _plan(ds, 1024, k=6)["token_tile"] == 64      # 6144 pairs over 160 experts
    assert _plan(ds, 1, k=6)["token_tile"] == 16
    # fine-grained experts (E >= 16 k): at least 32 rows from M = 32, where an uneven router
    # can give one expert several 16-row chunks; few experts keep the mean-based tile
    assert [_plan(ds, M, k=6)["token_tile"] for M in (16, 31, 32, 256, 512, 2048)] == [16, 16, 32, 32, 32, 128]
    assert _plan(dict(ds, E=95), 32, k=6)["token_tile"] == 16      # E < 16 k
    assert _plan(dict(ds, E=96), 32, k=6)["token_tile"] == 32
    assert _plan(ds, 256, k=6, token_tile=16)["token_tile"] == 16  # the option still decides
    assert _plan(MIXTRAL, 32)["token_tile"] == 16                  # E / k = 4
    with pytest.raises(q.QmoeError):
        q.qmoe_describe_plan(_layer_struct(**MIXTRAL), 16, 2, None, -1)


def test_header_is_plain_c99(tmp_path):
    """include/qmoe.h compiles as strict C99 (no C++ or torch types in the ABI), and its structs
    have the sizes the binding declares."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    src = tmp_path / "h.c"
    src.write_text('#include "qmoe.h"\n'
                   "typedef char a[sizeof(qmoe_options) == %d ? 1 : -1];\n"
                   "typedef char b[sizeof(qmoe_plan_info) == %d ? 1 : -1];\n"
                   "typedef char c[sizeof(qmoe_layer) == %d ? 1 : -1];\n"
                   "typedef char d[sizeof(qmoe_linear) == %d ? 1 : -1];\n"
                   % (ctypes.sizeof(N.QmoeOptions), ctypes.sizeof(N.QmoePlanInfo), ctypes.sizeof(N.QmoeLayer),
                      ctypes.sizeof(N.QmoeLinear)))
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc, "-c", str(src), "-o",
                        str(tmp_path / "h.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


# ----------------------------------------------------------------------------
# 2:4-sparse int8 and the dense linear layer
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("gs,act", [(-1, "bf16"), (128, "f16"), (128, "bf16")])
def test_pack_int8_24_round_trip_and_layout(gs, act):
    from synth import make_layer, to_u16_bits
    wl = Workload("t", 3, 2, 256, 384, "int8s24", gs, act, False, 0.0, (1,))
    L = make_layer(wl, seed=6)
    if gs == -1:
        pk = q.qmoe_pack_int8_24(3, 256, 384, "f32", L.q13, L.s13, L.q2, L.s2, -1)
        assert pk["w13"].nbytes == 3 * (768 // 128) * 2 * 10240
        q13, s13, q2, s2 = q.qmoe_unpack_int8_24(3, 256, 384, pk["w13"], pk["s13"], pk["w2"], pk["s2"], -1)
        assert np.array_equal(s13, L.s13) and np.array_equal(s2, L.s2)
    else:
        s13b, s2b = to_u16_bits(L.s13, act), to_u16_bits(L.s2, act)
        pk = q.qmoe_pack_int8_24(3, 256, 384, act, L.q13, s13b, L.q2, s2b, 128)
        assert pk["w13"].nbytes == 3 * (768 // 128) * 2 * 10496
        q13, s13, q2, s2 = q.qmoe_unpack_int8_24(3, 256, 384, pk["w13"], None, pk["w2"], None, 128)
        assert np.array_equal(s13, s13b) and np.array_equal(s2, s2b)
    assert np.array_equal(q13, L.q13) and np.array_equal(q2, L.q2)
    # documented layout of W2, expert 0, tile 0, K stage 0: row r, half h, group g:
    # kept codes at bytes (h*128 + r)*32 + 2g + {0,1}; positions in the sparse-MMA lane order at 8192
    blk = pk["w2"][:10240 if gs == -1 else 10496]
    for r in (0, 77, 8, 127):
        for h in (0, 1):
            for g in range(16):
                m = _sparse_position(blk[8192:10240], r, 16 * h + g)
                i0, i1 = m & 3, m >> 2
                assert i0 < i1
                c4 = L.q2[0, r, 64 * h + 4 * g: 64 * h + 4 * g + 4]
                v = blk[(h * 128 + r) * 32 + 2 * g: (h * 128 + r) * 32 + 2 * g + 2].view(np.int8)
                assert (v[0], v[1]) == (c4[i0], c4[i1])
                assert all(c4[i] == 0 for i in range(4) if i not in (i0, i1))


def test_pack_int8_24_rejects_three_of_four_and_minus_128():
    q13 = np.zeros((1, 256, 128), np.int8)
    q2 = np.zeros((1, 128, 128), np.int8)
    s13 = np.ones((1, 256), np.float32)
    s2 = np.ones((1, 128), np.float32)
    q13[0, 5, 8:11] = [1, 2, 3]
    with pytest.raises(q.QmoeError):
        q.qmoe_pack_int8_24(1, 128, 128, "f32", q13, s13, q2, s2, -1)
    q13[0, 5, 8:11] = [1, 0, 3]
    q2[0, 0, 0] = -128
    with pytest.raises(q.QmoeError):
        q.qmoe_pack_int8_24(1, 128, 128, "f32", q13, s13, q2, s2, -1)
    q2[0, 0, 0] = -127
    q.qmoe_pack_int8_24(1, 128, 128, "f32", q13, s13, q2, s2, -1)


LINEAR_FORMATS = [("int4", 128, "f16", True), ("int4", -1, "bf16", False), ("int4zp", 128, "bf16", True),
                  ("int4s24", 128, "f16", False), ("int8", -1, "bf16", False), ("int8g", 128, "f16", False),
                  ("int8s24", -1, "bf16", False), ("int8s24", 128, "f16", False)]


@pytest.mark.parametrize("qt,gs,act,ao", LINEAR_FORMATS)
def test_pack_linear_round_trip(qt, gs, act, ao):
    from synth import make_linear, to_u16_bits
    lin = make_linear(256, 384, qt, gs, act, act_order=ao, seed=2)
    pk = q.qmoe_pack_linear(qt, 256, 384, act, lin.q, lin.s, gs, lin.z, lin.g_idx)
    assert pk["w"].nbytes == q.packed_bytes(qt, 1, 256, 384, gs)
    res = q.qmoe_unpack_linear(qt, 256, 384, pk, gs, lin.g_idx)
    assert np.array_equal(res[0], lin.q)
    if lin.s.ndim == 1:
        assert np.array_equal(res[1], lin.s)
    else:
        assert np.array_equal(res[1], to_u16_bits(lin.s, act))
    if qt == "int4zp":
        assert np.array_equal(res[2], lin.z)
    if ao:
        p = pk["perm"]
        assert sorted(p.tolist()) == list(range(384)) and np.all(np.diff(lin.g_idx[p]) >= 0)


def test_linear_plan_and_validation_are_host_only():
    L = q.lib()
    ok = N.QmoeLinear(4096, 14336, 128, N.QMOE_INT4_GROUP, N.QMOE_F16, N.QMOE_F16, None, None, None)
    assert L.qmoe_linear_workspace_size(ctypes.byref(ok), 16, None) > 0
    p = q.qmoe_linear_describe_plan(ok, 16, num_sms=152)
    assert p["token_tile"] == 16 and p["issuers"] == 2 and p["split1"] >= 1 and p["split2"] == 0
    assert q.qmoe_linear_describe_plan(ok, 100, num_sms=152)["token_tile"] == 128
    for bad in (N.QmoeLinear(100, 128, 128, N.QMOE_INT4_GROUP, N.QMOE_F16, N.QMOE_F16, None, None, None),
                N.QmoeLinear(128, 128, 64, N.QMOE_INT4_GROUP, N.QMOE_F16, N.QMOE_F16, None, None, None),
                N.QmoeLinear(128, 128, -1, N.QMOE_INT8_24, N.QMOE_F16, N.QMOE_F16, None, None, None),
                N.QmoeLinear(128, 128, 128, 99, N.QMOE_F16, N.QMOE_F16, None, None, None)):
        assert L.qmoe_linear_workspace_size(ctypes.byref(bad), 16, None) == 0
        assert L.qmoe_linear_forward(ctypes.byref(bad), None, 16, None, None, 0, None, None) != q.QMOE_OK
    # a valid layer with no workspace: rejected before any device access
    assert L.qmoe_linear_forward(ctypes.byref(ok), None, 16, None, None, 0, None, None) == q.QMOE_ERR_WORKSPACE
    assert L.qmoe_linear_forward(ctypes.byref(ok), None, 0, None, None, 0, None, None) == q.QMOE_OK
