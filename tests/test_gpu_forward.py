"""The fused layer on the GPU (through the C ABI) against the float64 oracle.

Shapes are small enough for the oracle to finish in seconds yet span several
128-row weight tiles, several 128-wide K stages, ragged token chunks, split-K
and multi-chunk experts.
"""
import copy

import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_moe_gb300 as q
from synth import Inputs, Workload, make_inputs, make_layer, round_to
from tests.gpu_util import assert_parity, device_inputs, device_layer, ensure_built, run_forward

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _wl(qt="int4", act="f16", act_order=False, E=8, k=2, H=384, I=256, zipf=0.0, gs=None):
    if gs is None:
        gs = -1 if qt == "int8" else 128
    return Workload(f"t_{qt}_{act}_{act_order}_{gs}", E, k, H, I, qt, gs, act, act_order, zipf, (1,))


_LAYERS = {}


def _layer(wl, seed=0):
    key = (wl, seed)
    if key not in _LAYERS:
        L = make_layer(wl, seed=seed)
        _LAYERS[key] = (L, device_layer(L))
    return _LAYERS[key]


def _check(wl, M, seed=0, opts=None, inp=None, what=""):
    L, dl = _layer(wl)
    if inp is None:
        inp = make_inputs(wl, M, seed=seed + 10)
    x, ids, w = device_inputs(wl, inp)
    out, _ = run_forward(dl, x, ids, w, opts=opts)
    got = out.float().cpu().numpy()
    ref = oracle.moe_forward(L, inp.x, inp.topk_ids, inp.topk_weights)
    return assert_parity(got, ref, what or f"{wl.name} M={M}")


VARIANTS = [("int4", "f16", False), ("int4", "bf16", False), ("int4", "f16", True), ("int4", "bf16", True),
            ("int8", "bf16", False), ("int8", "f16", False)]
# weight formats beyond the pages' two: per-group zero points, channel-wise int4, group-128 int8
OTHER_FORMATS = [("int4zp", "f16", False, 128), ("int4zp", "bf16", True, 128), ("int4zp", "bf16", False, -1),
                 ("int4", "f16", False, -1), ("int4", "bf16", False, -1), ("int8g", "f16", False, 128),
                 ("int8g", "bf16", False, 128), ("int4s24", "f16", False, 128), ("int4s24", "bf16", False, 128),
                 ("int4s24", "f16", False, -1), ("int8s24", "bf16", False, -1), ("int8s24", "f16", False, 128),
                 ("int8s24", "bf16", False, 128)]


@pytest.mark.parametrize("qt,act,ao", VARIANTS)
@pytest.mark.parametrize("M", [1, 7, 64, 129])
def test_forward_parity(qt, act, ao, M):
    _check(_wl(qt, act, ao), M)


@pytest.mark.parametrize("qt,act,ao,gs", OTHER_FORMATS)
@pytest.mark.parametrize("M", [1, 40, 129])
def test_forward_parity_other_formats(qt, act, ao, gs, M):
    _check(_wl(qt, act, ao, gs=gs), M)


@pytest.mark.parametrize("qt,act,ao,gs", OTHER_FORMATS[:2] + OTHER_FORMATS[5:6] + OTHER_FORMATS[7:8] + OTHER_FORMATS[10:12])
@pytest.mark.parametrize("split1,split2,tile", [(3, 2, 0), (2, 1, 16), (1, 2, 128)])
def test_forward_other_formats_forced_split_and_tile(qt, act, ao, gs, split1, split2, tile):
    _check(_wl(qt, act, ao, gs=gs), 40, opts=q.make_options(split1, split2, tile))


@pytest.mark.parametrize("qt,act,ao", VARIANTS[:1] + VARIANTS[3:5])
@pytest.mark.parametrize("split1,split2,tile", [(3, 2, 0), (2, 1, 16), (1, 2, 128), (3, 2, 32)])
def test_forward_forced_split_and_tile(qt, act, ao, split1, split2, tile):
    _check(_wl(qt, act, ao), 40, opts=q.make_options(split1, split2, tile))


@pytest.mark.parametrize("qt,act,ao,gs", [("int4", "f16", False, 128), ("int4", "bf16", True, 128),
                                          ("int4zp", "bf16", False, 128), ("int8", "bf16", False, -1),
                                          ("int8g", "f16", False, 128), ("int4s24", "f16", False, 128),
                                          ("int8s24", "bf16", False, -1)])
@pytest.mark.parametrize("M,split1,split2,tile", [(1, 0, 0, 0), (40, 0, 0, 0), (129, 0, 0, 0), (40, 3, 2, 0),
                                                  (300, 1, 1, 128), (40, 2, 1, 64)])
def test_forward_two_dequant_sets(qt, act, ao, gs, M, split1, split2, tile):
    """The GEMMs with two dequant sets of eight half-row warps (the default is four
    sets of four whole-row warps wherever the rings allow it), every tile size."""
    _check(_wl(qt, act, ao, gs=gs), M, opts=q.make_options(split1, split2, tile, dq_sets=2))


@pytest.mark.parametrize("qt,act,ao,gs", [("int4", "f16", False, 128), ("int4", "bf16", True, 128),
                                          ("int8", "bf16", False, -1), ("int4zp", "f16", False, 128),
                                          ("int4s24", "f16", False, 128), ("int8s24", "bf16", False, -1)])
@pytest.mark.parametrize("M,split1,split2,tile", [(300, 0, 0, 192), (1200, 0, 0, 256), (1200, 0, 0, 192),
                                                  (1200, 2, 1, 256), (129, 0, 0, 144), (1100, 0, 0, 208)])
def test_forward_large_token_tiles(qt, act, ao, gs, M, split1, split2, tile):
    """Token tiles above 128 rows (MMA N up to 256): one issuer, a two-slot A
    ring, and a single accumulator buffer where two do not fit tensor memory."""
    _check(_wl(qt, act, ao, gs=gs), M, opts=q.make_options(split1, split2, tile))


@pytest.mark.parametrize("qt,act,ao,gs", [("int4", "f16", False, 128), ("int4", "bf16", True, 128),
                                          ("int4", "bf16", False, -1), ("int8", "bf16", False, -1),
                                          ("int8", "f16", False, -1)])
@pytest.mark.parametrize("M,split1,split2,tile", [(1, 0, 0, 0), (7, 0, 0, 0), (40, 0, 0, 0), (129, 0, 0, 0),
                                                  (40, 3, 2, 0), (300, 1, 1, 128), (40, 2, 1, 64), (129, 0, 0, 32),
                                                  (1200, 0, 0, 128), (300, 0, 0, 256)])
def test_forward_cta_pairs(qt, act, ao, gs, M, split1, split2, tile):
    """The GEMMs on CTA pairs: M = 256 MMAs over two SMs, each CTA with half of
    every token tile; the down GEMM's 3 weight tiles (H = 384) leave the last
    pair's odd CTA a phantom that computes and stores nothing of its own."""
    _check(_wl(qt, act, ao, gs=gs), M, opts=q.make_options(split1, split2, tile, cta_pair=1))


@pytest.mark.parametrize("M,tile,ring,sets", [(40, 64, 1, 0), (129, 128, 0, 2), (300, 64, 2, 0), (7, 16, 1, 2)])
def test_forward_cta_pairs_rings(M, tile, ring, sets):
    """CTA pairs with a token-tile ring of one or two A-ring depths and with two
    dequant sets."""
    _check(_wl("int4", "f16", False), M, opts=q.make_options(0, 0, tile, token_ring=ring, dq_sets=sets, cta_pair=1))


@pytest.mark.parametrize("act,ao,gs", [("f16", False, 128), ("bf16", True, 128), ("f16", False, -1), ("bf16", False, -1)])
@pytest.mark.parametrize("M,split1,split2", [(1, 0, 0), (7, 0, 0), (40, 0, 0), (40, 3, 2), (16, 1, 1), (33, 2, 2)])
@pytest.mark.parametrize("epi", [1, 2])
def test_int4_group_epilogue_on_and_off(act, ao, gs, M, split1, split2, epi):
    """Symmetric int4 at 16-row token tiles with the per-group fp32 scaling epilogue
    (raw magic-number A, tokens pre-divided by 16 at the x16 positions, per-stage
    TMEM sums) and without it."""
    _check(_wl("int4", act, ao, gs=gs), M, opts=q.make_options(split1, split2, 16, int4_group_epilogue=epi))


@pytest.mark.parametrize("M,ring,sets", [(1, 1, 0), (40, 1, 0), (40, 2, 2), (7, 2, 2), (33, 1, 2)])
def test_int4_group_epilogue_rings(M, ring, sets):
    """The per-group scaling epilogue with a token-tile ring of one A-ring depth
    (its D slots then come back through the same "done" barriers as the token
    tiles) and with two dequant sets of half-row warps."""
    _check(_wl("int4", "f16", False, gs=128), M,
           opts=q.make_options(0, 0, 16, token_ring=ring, dq_sets=sets, int4_group_epilogue=1))


@pytest.mark.parametrize("qt,act", [("int8", "f16"), ("int8", "bf16")])
def test_int8_token_tile_128_single_accumulator_per_issuer(qt, act):
    # 128-row chunks: each MMA issuer has one TMEM accumulator, summed by the epilogue
    _check(_wl(qt, act), 300, opts=q.make_options(0, 0, 128))


@pytest.mark.parametrize("qt,act", [("int4", "bf16"), ("int4", "f16"), ("int8", "bf16"), ("int8", "f16")])
def test_token_tile_limits_rejected(qt, act):
    # token tiles up to 256 rows; TMEM (512 columns) holds one fp32 accumulator of the
    # token tile per MMA issuer plus the A slots, so two issuers of 256 rows do not fit
    wl = _wl(qt, act)
    _, dl = _layer(wl)
    for opts in (q.make_options(0, 0, 272), q.make_options(0, 0, 256, issuers=2)):
        with pytest.raises(q.QmoeError) as ei:
            q.qmoe_workspace_size(dl, 40, 2, opts)
        assert ei.value.status == q.QMOE_ERR_INVALID_ARG


@pytest.mark.parametrize("qt,act,ao,exps,spread", [("int4", "bf16", False, (24, -24), 8),
                                                    ("int4", "bf16", True, (16, -20), 8),
                                                    ("int8", "bf16", False, (30, -30), 8),
                                                    ("int4", "f16", False, (0,), 4),
                                                    ("int8", "f16", False, (-2,), 4)])
def test_activation_magnitudes(qt, act, ao, exps, spread):
    """Both GEMMs run in f16 on rows scaled by powers of two: bf16 inputs far
    outside f16's range, and rows of very different magnitude, keep the bar per
    row.  (f16 layers stay where their f16 output is representable.)"""
    wl = _wl(qt, act, ao)
    L, dl = _layer(wl)
    M = 48
    base = make_inputs(wl, M, seed=31)
    rng = np.random.default_rng(7)
    for ex in exps:
        # every row scaled by 2^ex and rows spread over a further 2^-spread .. 2^spread
        row_e = ex + rng.integers(-spread, spread + 1, size=(M, 1))
        x = round_to(np.ldexp(base.x.astype(np.float64), row_e), act).astype(np.float32)
        inp = Inputs(x, base.topk_ids, base.topk_weights, base.logits)
        xd, ids, w = device_inputs(wl, inp)
        out, _ = run_forward(dl, xd, ids, w)
        got = out.float().cpu().numpy()
        ref = oracle.moe_forward(L, inp.x, inp.topk_ids, inp.topk_weights)
        assert np.isfinite(got).all()
        for m in range(M):
            assert_parity(got[m:m + 1], ref[m:m + 1], f"{wl.name} 2^{ex} row {m}")


def test_bf16_rows_near_the_top_of_the_range():
    """bf16 rows whose largest magnitude is ~2^118 (bf16 reaches 2^128): the
    power-of-two row scaling must bring them into f16 range.  Per-column int8
    applies its fp32 scale to the accumulator, so W13 scales of ~2^-123 keep
    the layer's values finite: h = 16 * (x . W)."""
    wl = _wl("int8", "bf16")
    L0, _ = _layer(wl)
    L = copy.copy(L0)
    L.s13 = (L0.s13.astype(np.float64) * 2.0 ** -112).astype(np.float32)
    dl = device_layer(L)
    M = 24
    base = make_inputs(wl, M, seed=41)
    x = round_to(np.ldexp(base.x.astype(np.float64), 116), "bf16").astype(np.float32)
    inp = Inputs(x, base.topk_ids, base.topk_weights, base.logits)
    xd, ids, w = device_inputs(wl, inp)
    out, _ = run_forward(dl, xd, ids, w)
    got = out.float().cpu().numpy()
    ref = oracle.moe_forward(L, inp.x, inp.topk_ids, inp.topk_weights)
    assert np.isfinite(got).all()
    for m in range(M):
        assert_parity(got[m:m + 1], ref[m:m + 1], f"bf16 2^116 row {m}")


def test_multi_chunk_expert_and_empty_experts():
    wl = _wl("int4", "bf16")
    M = 300
    base = make_inputs(wl, M, seed=21)
    ids = base.topk_ids.copy()
    ids[:, 0] = 3                          # expert 3 takes every token -> several chunks
    ids[:, 1] = np.where(ids[:, 1] == 3, 5, ids[:, 1])
    ids[::7, 1] = 6
    inp = Inputs(base.x, ids.astype(np.int32), base.topk_weights, base.logits)
    _check(wl, M, inp=inp, what="one hot expert")


def test_many_experts_topk6_skewed():
    wl = _wl("int8", "bf16", E=160, k=6, H=256, I=256, zipf=1.1)
    for M in (1, 5, 96):
        _check(wl, M)


def test_many_experts_int4_actorder():
    wl = _wl("int4", "f16", True, E=64, k=4, H=256, I=384)
    _check(wl, 33)


def test_deterministic_and_host_path_identical():
    wl = _wl("int4", "f16", True)
    L, dl = _layer(wl)
    inp = make_inputs(wl, 50, seed=5)
    x, ids, w = device_inputs(wl, inp)
    a, _ = run_forward(dl, x, ids, w)
    b, _ = run_forward(dl, x, ids, w)
    assert torch.equal(a, b)
    xh = x.cpu().pin_memory()
    idsh = ids.cpu().pin_memory()
    wh = w.cpu().pin_memory()
    outh = torch.empty_like(xh).pin_memory()
    ws = q.alloc_workspace(q.qmoe_workspace_size_host(dl, 50, wl.k))
    q.qmoe_forward_host(dl, xh, idsh, wh, outh, ws)
    torch.cuda.synchronize()
    assert q.qmoe_read_device_status(ws) == q.QMOE_OK
    assert torch.equal(outh, a.cpu())


def _offset_pinned(t, offset_bytes):
    """A pinned copy of t whose data starts offset_bytes past a pinned allocation's start."""
    n = t.numel() * t.element_size()
    raw = torch.empty(n + offset_bytes, dtype=torch.uint8).pin_memory()
    view = raw[offset_bytes:offset_bytes + n].view(t.dtype).view(t.shape)
    view.copy_(t)
    return view


@pytest.mark.parametrize("memory", ["pinned", "pageable", "pinned_unaligned"])
@pytest.mark.parametrize("M", [1, 50, 300])
def test_host_path_memory_kinds(memory, M):
    """qmoe_forward_host with page-locked mapped buffers (the kernels read the
    inputs and write out in host memory in place), with pageable buffers and
    with pinned buffers whose x and out miss the 256-byte alignment (both staged
    through device copies): all bit-identical to the device-buffer forward."""
    wl = _wl("int4", "bf16", False)
    L, dl = _layer(wl)
    inp = make_inputs(wl, M, seed=9)
    x, ids, w = device_inputs(wl, inp)
    want, _ = run_forward(dl, x, ids, w)
    if memory == "pinned":
        xh, idsh, wh = x.cpu().pin_memory(), ids.cpu().pin_memory(), w.cpu().pin_memory()
        outh = torch.full_like(xh, float("nan")).pin_memory()
    elif memory == "pageable":
        xh, idsh, wh = x.cpu(), ids.cpu(), w.cpu()
        outh = torch.full_like(xh, float("nan"))
    else:
        xh, idsh, wh = _offset_pinned(x.cpu(), 16), ids.cpu().pin_memory(), w.cpu().pin_memory()
        outh = _offset_pinned(torch.full_like(x.cpu(), float("nan")), 16)
    ws = q.alloc_workspace(q.qmoe_workspace_size_host(dl, M, wl.k))
    for _ in range(2):
        q.qmoe_forward_host(dl, xh, idsh, wh, outh, ws)
        torch.cuda.synchronize()
        assert q.qmoe_read_device_status(ws) == q.QMOE_OK
        assert torch.equal(outh, want.cpu()), memory
    # the host rewrites its buffers in place between calls (a serving loop): the
    # next call must see the new contents, not data cached from the last one
    inp2 = make_inputs(wl, M, seed=19)
    x2, ids2, w2 = device_inputs(wl, inp2)
    want2, _ = run_forward(dl, x2, ids2, w2)
    xh.copy_(x2.cpu())
    idsh.copy_(ids2.cpu())
    wh.copy_(w2.cpu())
    q.qmoe_forward_host(dl, xh, idsh, wh, outh, ws)
    torch.cuda.synchronize()
    assert torch.equal(outh, want2.cpu()), memory + " after rewriting the host inputs"


def test_zero_tokens_is_a_no_op():
    wl = _wl()
    _, dl = _layer(wl)
    x = torch.empty((0, wl.H), dtype=torch.float16, device="cuda")
    ids = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    w = torch.empty((0, 2), dtype=torch.float32, device="cuda")
    out = q.qmoe_forward(dl, x, ids, w, workspace=q.alloc_workspace(256))
    assert out.shape == (0, wl.H)


def test_bad_expert_id_is_reported_and_dropped():
    wl = _wl()
    L, dl = _layer(wl)
    inp = make_inputs(wl, 6, seed=8)
    ids = inp.topk_ids.copy()
    ids[2, 1] = 99
    x, dids, w = device_inputs(wl, Inputs(inp.x, ids, inp.topk_weights, inp.logits))
    out, st = run_forward(dl, x, dids, w, check_status=False)
    assert st == q.QMOE_ERR_BAD_EXPERT_ID
    wts = inp.topk_weights.copy()
    wts[2, 1] = 0.0
    ids_ok = ids.copy()
    ids_ok[2, 1] = 0
    ref = oracle.moe_forward(L, inp.x, ids_ok, wts)
    assert_parity(out.float().cpu().numpy(), ref, "bad id dropped")


@pytest.mark.parametrize("qt,act,ao", [("int4", "f16", False), ("int4", "bf16", True), ("int8", "bf16", False),
                                      ("int4s24", "f16", False)])
@pytest.mark.parametrize("M,split2", [(1, 0), (7, 0), (40, 0), (40, 2), (129, 1), (129, 0), (600, 0)])
def test_topk_reduce_in_gemm_bit_identical(qt, act, ao, M, split2):
    """The top-k reduction in the down GEMM's epilogue (arrival counters, last
    warp sums) and the separate reduce kernel sum in the same order: outputs are
    bit-identical, and match the oracle."""
    wl = _wl(qt, act, ao)
    L, dl = _layer(wl)
    inp = make_inputs(wl, M, seed=21)
    x, ids, w = device_inputs(wl, inp)
    outs = []
    for mode in (1, 2):
        out, _ = run_forward(dl, x, ids, w, opts=q.make_options(0, split2, topk_reduce=mode))
        outs.append(out.float().cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
    assert_parity(outs[0], oracle.moe_forward(L, inp.x, inp.topk_ids, inp.topk_weights), f"{wl.name} M={M}")


@pytest.mark.parametrize("mode", [1, 2])
def test_token_without_valid_expert_is_zero(mode):
    """A token all of whose top-k ids are invalid has no pair in any GEMM item:
    its output row is zero on both reduction paths (status reports the bad ids)."""
    wl = _wl()
    L, dl = _layer(wl)
    inp = make_inputs(wl, 9, seed=4)
    ids = inp.topk_ids.copy()
    ids[3, :] = -1
    ids[5, 0] = 1000
    x, dids, w = device_inputs(wl, Inputs(inp.x, ids, inp.topk_weights, inp.logits))
    out, st = run_forward(dl, x, dids, w, opts=q.make_options(topk_reduce=mode), check_status=False)
    assert st == q.QMOE_ERR_BAD_EXPERT_ID
    got = out.float().cpu().numpy()
    assert np.all(got[3] == 0.0)
    wts = inp.topk_weights.copy()
    wts[3, :] = 0.0
    wts[5, 0] = 0.0
    ids_ok = np.where(ids < 0, 0, np.where(ids >= wl.E, 0, ids)).astype(ids.dtype)
    assert_parity(got, oracle.moe_forward(L, inp.x, ids_ok, wts), "invalid ids dropped")


def test_rejects_wrong_device_pointer_and_small_workspace():
    wl = _wl()
    _, dl = _layer(wl)
    inp = make_inputs(wl, 4, seed=1)
    x, ids, w = device_inputs(wl, inp)
    ws = q.alloc_workspace(q.qmoe_workspace_size(dl, 4, 2) - 1024)
    with pytest.raises(q.QmoeError) as ei:
        q.qmoe_forward(dl, x, ids, w, workspace=ws)
    assert ei.value.status == q.QMOE_ERR_WORKSPACE
    ws = q.alloc_workspace(q.qmoe_workspace_size(dl, 4, 2))
    with pytest.raises(q.QmoeError) as ei:
        q.qmoe_forward(dl, x.cpu(), ids, w, workspace=ws)
    assert ei.value.status == q.QMOE_ERR_DEVICE_MISMATCH
