"""Full-size parity: every benchmark workload at every batch size it is measured
at, launched as bench.py launches it (default plan), checked element by element
against the oracle on at least 16 tokens of each batch.

Tokens are independent rows of the layer, so the oracle computes only the
sampled ones, each expert dequantized once per workload for all its batch
sizes.  The sample covers, for every expert that received pairs, the token of
the first row of its first chunk and of the first and last rows of its last
(possibly partial) chunk (a chunk is up to token-tile rows of one expert's
pairs, in ascending pair order), plus seeded random tokens.  Every output
element of every token is also checked to be finite.
"""
import gc
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_moe_gb300 as q
from synth import WORKLOADS, Workload, make_inputs, make_layer
from tests.gpu_util import assert_parity, device_inputs, device_layer, ensure_built, run_forward

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# every (workload, M) the benchmark reports
FULL_WORKLOADS = ("mixtral8x7b_w4", "mixtral8x7b_w4_actorder", "mixtral8x7b_w8", "deepseekv2_w8",
                  "mixtral8x22b_w4", "mixtral8x7b_w4s24", "mixtral8x7b_w8s24")
FULL = [(name, M) for name in FULL_WORKLOADS for M in WORKLOADS[name].Ms]

# the Mixtral-8x7B shape in the other weight formats (zero points, group-128 int8)
WORKLOADS_OTHER = {
    "mixtral8x7b_w4zp": Workload("mixtral8x7b_w4zp", 8, 2, 4096, 14336, "int4zp", 128, "bf16", False, 0.0, (16,)),
    "mixtral8x7b_w8g": Workload("mixtral8x7b_w8g", 8, 2, 4096, 14336, "int8g", 128, "f16", False, 0.0, (16,)),
}
MIN_ROWS = 16


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def chunk_boundary_tokens(topk_ids: np.ndarray, T: int) -> list:
    """Tokens of the first row of each expert's first chunk and of the first and
    last rows of its last chunk (rows of an expert are its pairs p = m*k + j in
    ascending order, T rows per chunk)."""
    k = topk_ids.shape[1]
    flat = topk_ids.reshape(-1)
    toks = []
    for e in np.unique(flat):
        pairs = np.nonzero(flat == e)[0]
        last0 = (pairs.size - 1) // T * T
        toks += [int(pairs[0]) // k, int(pairs[last0]) // k, int(pairs[-1]) // k]
    return toks


def sample_tokens(topk_ids: np.ndarray, T: int, seed: int, n_min: int = MIN_ROWS, n_random: int = 4) -> list:
    M = topk_ids.shape[0]
    rows = list(dict.fromkeys(chunk_boundary_tokens(topk_ids, T)))
    want = min(M, max(n_min, len(rows) + n_random))
    for m in np.random.default_rng(seed).permutation(M):
        if len(rows) >= want:
            break
        if int(m) not in rows:
            rows.append(int(m))
    return rows


def _oracle_rows(layer, batches):
    """The oracle on the sampled rows of every batch; experts are split over a few
    threads (each dequantizes its own experts) and the partial outputs summed."""
    E = layer.wl.E
    n = max(1, min(4, (os.cpu_count() or 1) // 4, E))
    groups = [list(range(g, E, n)) for g in range(n)]
    if n == 1:
        return oracle.moe_forward_batches(layer, batches)
    with ThreadPoolExecutor(n) as ex:
        parts = list(ex.map(lambda g: oracle.moe_forward_batches(layer, batches, experts=g), groups))
    return [sum(p[i] for p in parts) for i in range(len(batches))]


_RESULTS = {}


def _results(name):
    """Run every batch size of a workload on the GPU, then the oracle on the sampled tokens."""
    if name in _RESULTS:
        return _RESULTS[name]
    _RESULTS.clear()
    gc.collect()
    torch.cuda.empty_cache()
    wl = WORKLOADS[name]
    L = make_layer(wl, seed=0)
    dl = device_layer(L)
    res, batches = {}, []
    for M in wl.Ms:
        inp = make_inputs(wl, M, seed=0)
        x, ids, w = device_inputs(wl, inp)
        out, _ = run_forward(dl, x, ids, w)
        got = out.float().cpu().numpy()
        T = q.qmoe_describe_plan(dl, M, wl.k)["token_tile"]
        rows = sample_tokens(inp.topk_ids, T, seed=M)
        res[M] = {"got": got[rows], "finite": bool(np.isfinite(got).all()), "rows": rows, "T": T}
        batches.append((inp.x, inp.topk_ids, inp.topk_weights, rows))
        del x, ids, w, out, got
        torch.cuda.empty_cache()
    del dl
    torch.cuda.empty_cache()
    for M, ref in zip(wl.Ms, _oracle_rows(L, batches)):
        res[M]["ref"] = ref
    del L
    gc.collect()
    _RESULTS[name] = res
    return res


@pytest.mark.parametrize("name,M", FULL)
def test_full_size_parity(name, M):
    r = _results(name)[M]
    assert r["finite"], f"{name} M={M}: non-finite output"
    assert len(r["rows"]) >= min(M, MIN_ROWS)
    assert_parity(r["got"], r["ref"], f"{name} M={M} T={r['T']} rows={r['rows'][:24]}")


_cache = {}


def _layer(name):
    if name not in _cache:
        _cache.clear()
        _RESULTS.clear()
        gc.collect()
        torch.cuda.empty_cache()
        L = make_layer(WORKLOADS.get(name) or WORKLOADS_OTHER[name], seed=0)
        _cache[name] = (L, device_layer(L))
    return _cache[name]


@pytest.mark.parametrize("name", sorted(WORKLOADS_OTHER))
def test_full_size_other_formats(name):
    wl = WORKLOADS_OTHER[name]
    L, dl = _layer(name)
    M = 16
    inp = make_inputs(wl, M, seed=0)
    x, ids, w = device_inputs(wl, inp)
    out, _ = run_forward(dl, x, ids, w)
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    rows = sample_tokens(inp.topk_ids, q.qmoe_describe_plan(dl, M, wl.k)["token_tile"], seed=3, n_min=4,
                         n_random=0)[:6]
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
