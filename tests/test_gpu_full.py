"""Full-size parity: every benchmark workload at its full shape, launched as
bench.py launches it (default plan), checked on sampled tokens that the
oracle computes one by one (tokens are independent rows of the layer)."""
import gc

import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_moe_gb300 as q
from synth import WORKLOADS, Workload, make_inputs, make_layer
from tests.gpu_util import assert_parity, device_inputs, device_layer, ensure_built, run_forward

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# the Mixtral-8x7B shape in the other weight formats (zero points, group-128 int8)
WORKLOADS_OTHER = {
    "mixtral8x7b_w4zp": Workload("mixtral8x7b_w4zp", 8, 2, 4096, 14336, "int4zp", 128, "bf16", False, 0.0, (16,)),
    "mixtral8x7b_w8g": Workload("mixtral8x7b_w8g", 8, 2, 4096, 14336, "int8g", 128, "f16", False, 0.0, (16,)),
}

# (workload, M, number of sampled tokens)
CASES = [
    ("mixtral8x7b_w4zp", 16, 2),
    ("mixtral8x7b_w8g", 16, 2),
    ("mixtral8x7b_w4s24", 16, 2),
    ("mixtral8x7b_w4", 16, 4),
    ("mixtral8x7b_w4", 1, 1),
    ("mixtral8x7b_w4_actorder", 16, 3),
    ("mixtral8x7b_w8", 128, 3),
    ("deepseekv2_w8", 256, 3),
    ("mixtral8x22b_w4", 2048, 2),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


_cache = {}


def _layer(name):
    if name not in _cache:
        _cache.clear()
        gc.collect()
        torch.cuda.empty_cache()
        L = make_layer(WORKLOADS.get(name) or WORKLOADS_OTHER[name], seed=0)
        _cache[name] = (L, device_layer(L))
    return _cache[name]


@pytest.mark.parametrize("name,M,n_sample", CASES)
def test_full_size_sampled(name, M, n_sample):
    wl = WORKLOADS.get(name) or WORKLOADS_OTHER[name]
    L, dl = _layer(name)
    inp = make_inputs(wl, M, seed=0)
    x, ids, w = device_inputs(wl, inp)
    out, _ = run_forward(dl, x, ids, w)
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    # sample tokens whose experts overlap, so the oracle dequantizes few experts
    rng = np.random.default_rng(M)
    first = int(rng.integers(M))
    rows = [first]
    want = set(inp.topk_ids[first].tolist())
    for m in rng.permutation(M):
        if len(rows) >= n_sample:
            break
        if int(m) not in rows and len(want | set(inp.topk_ids[m].tolist())) <= len(want) + wl.k // 2:
            rows.append(int(m))
            want |= set(inp.topk_ids[m].tolist())
    for m in rng.permutation(M):
        if len(rows) >= n_sample:
            break
        if int(m) not in rows:
            rows.append(int(m))
    ref = oracle.moe_forward_rows(L, inp.x, inp.topk_ids, inp.topk_weights, rows)
    assert_parity(got[rows], ref, f"{name} M={M} rows={rows}")


def test_full_size_long_items_repeated():
    """Whole-K work items (no split) at decode size: every CTA runs hundreds of
    pipeline stages through the even/odd producer, dequant and MMA roles.
    Repeated runs on a NaN-filled workspace catch ordering faults that only
    show under some interleavings."""
    name, M = "mixtral8x7b_w4", 16
    wl = WORKLOADS[name]
    L, dl = _layer(name)
    inp = make_inputs(wl, M, seed=0)
    x, ids, w = device_inputs(wl, inp)
    rows = [0, 5, 11]
    ref = oracle.moe_forward_rows(L, inp.x, inp.topk_ids, inp.topk_weights, rows)
    first = None
    for rep in range(6):
        out, _ = run_forward(dl, x, ids, w, opts=q.make_options(1, 1))
        got = out.float().cpu().numpy()
        assert_parity(got[rows], ref, f"{name} M={M} split 1 rep {rep}")
        if first is None:
            first = got
        else:
            assert np.array_equal(first, got), "whole-K forward not bit-reproducible"
