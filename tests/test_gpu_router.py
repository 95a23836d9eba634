"""The top-k router on the GPU (through the C ABI) against the oracle: expert
ids bit-exact, weights within fp32 rounding; and the router-then-layer entry
point against the oracle router followed by the oracle layer."""
import math

import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_moe_gb300 as q
from synth import Workload, make_inputs, make_layer, round_to
from tests.gpu_util import assert_parity, device_inputs, device_layer, ensure_built

pytestmark = pytest.mark.gpu

_TD = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _logits(rng, M, E, kind, dt):
    if kind == "normal":
        lg = rng.standard_normal((M, E))
    elif kind == "ties":
        lg = rng.integers(-4, 5, size=(M, E)) * 0.5
    elif kind == "zipf":
        rank = rng.permutation(E) + 1
        lg = rng.standard_normal((M, E)) - 1.1 * np.log(rank)[None, :]
    else:  # masked: some -inf entries and one fully masked row
        lg = rng.standard_normal((M, E))
        lg[rng.random((M, E)) < 0.3] = -np.inf
        lg[0] = -np.inf
    lg = lg.astype(np.float32)
    if dt != "f32":
        lg = np.where(np.isfinite(lg), round_to(lg, dt), lg).astype(np.float32)
    return lg


def _run(lg, dt, k, renorm):
    t = torch.from_numpy(lg).to(_TD[dt]).cuda()
    ids, w = q.qmoe_route_topk(t, k, renorm)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("E,k", [(8, 2), (60, 4), (160, 6), (1024, 8), (64, 32), (5, 5)])
@pytest.mark.parametrize("kind", ["normal", "ties", "zipf", "masked"])
def test_router_parity(dt, E, k, kind):
    rng = np.random.default_rng(E * 31 + k)
    lg = _logits(rng, 67, E, kind, dt)
    for renorm in (True, False):
        ids, w = _run(lg, dt, k, renorm)
        rids, rw = oracle.route_topk(lg, k, renorm)
        assert np.array_equal(ids, rids), f"{dt} E={E} k={k} {kind} renorm={renorm}"
        # fp32 softmax: exp and the normalising sum (up to E terms) round
        np.testing.assert_allclose(w, rw, rtol=2e-6 * max(1, E // 32), atol=1e-7)


def test_router_large_batch_and_edge_cases():
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((5000, 160)).astype(np.float32)
    ids, w = _run(lg, "f32", 6, True)
    rids, rw = oracle.route_topk(lg[:200], 6, True)
    assert np.array_equal(ids[:200], rids)
    np.testing.assert_allclose(w[:200], rw, rtol=2e-6, atol=1e-7)
    assert np.all(np.abs(w.sum(axis=1) - 1.0) < 1e-5)
    t = torch.zeros((0, 8), dtype=torch.float32, device="cuda")
    q.qmoe_route_topk(t, 2)  # M = 0 launches nothing
    t = torch.zeros((4, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmoeError) as ei:
        q.qmoe_route_topk(t, 33)
    assert ei.value.status == q.QMOE_ERR_UNSUPPORTED
    with pytest.raises(q.QmoeError) as ei:
        q.qmoe_route_topk(torch.zeros((4, 8), dtype=torch.float32, device="cuda"), 9)
    assert ei.value.status == q.QMOE_ERR_INVALID_ARG


@pytest.mark.parametrize("qt,act,E,k,ldt", [("int4", "f16", 8, 2, "f32"), ("int8", "bf16", 16, 4, "bf16"),
                                             ("int4", "bf16", 12, 3, "f16")])
def test_forward_logits_parity(qt, act, E, k, ldt):
    wl = Workload(f"r_{qt}_{act}", E, k, 256, 256, qt, 128 if qt == "int4" else -1, act, False, 0.0, (1,))
    L = make_layer(wl, seed=3)
    dl = device_layer(L)
    M = 37
    inp = make_inputs(wl, M, seed=4)
    rng = np.random.default_rng(9)
    lg = _logits(rng, M, E, "normal", ldt)
    x, _, _ = device_inputs(wl, inp)
    out = q.qmoe_forward_logits(dl, x, torch.from_numpy(lg).to(_TD[ldt]).cuda(), k, True)
    rids, rw = oracle.route_topk(lg, k, True)
    ref = oracle.moe_forward(L, inp.x, rids, rw)
    assert_parity(out.float().cpu().numpy(), ref, f"{qt} {act} router+layer")
