"""moe_align_block_size on the GPU, bit-exact against the oracle (through the C ABI)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_moe_gb300 as q
from tests.gpu_util import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _check(ids_np, E, B, capacity=None):
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, np.int32)).cuda()
    s, ex, n = q.qmoe_moe_align(ids, E, B, capacity)
    torch.cuda.synchronize()
    rs, rex, rn = oracle.moe_align(ids_np, E, B, capacity)
    assert int(n.item()) == rn
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(ex.cpu().numpy(), rex)


def test_golden_examples():
    with open(os.path.join(os.path.dirname(__file__), "golden", "moe_align_examples.json")) as f:
        for c in json.load(f)["cases"]:
            _check(np.array(c["topk_ids"], np.int32), c["E"], c["block"])


@pytest.mark.parametrize("M,k,E,B", [
    (1, 2, 8, 16), (3, 2, 8, 16), (16, 2, 8, 16), (64, 2, 8, 16), (512, 2, 8, 16), (8192, 2, 8, 16),
    (1, 6, 160, 16), (1024, 6, 160, 16), (33, 4, 16, 1), (100, 2, 8, 256), (777, 3, 1024, 64), (5, 8, 8, 32),
])
def test_random_ids(M, k, E, B):
    rng = np.random.default_rng(M * 7 + E)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(M)]) if k <= E else rng.integers(0, E, (M, k))
    _check(ids, E, B)


def test_skewed_all_to_one_expert():
    ids = np.full((3000, 2), 5, np.int32)
    ids[:, 1] = 6
    ids[17, 0] = 0
    _check(ids, 8, 16)


def test_larger_capacity_and_empty():
    rng = np.random.default_rng(3)
    ids = rng.integers(0, 8, (10, 2)).astype(np.int32)
    _check(ids, 8, 16, capacity=10 * 2 + 8 * 15 + 37)
    _check(np.zeros((0, 2), np.int32), 8, 16)


def test_bad_ids_are_dropped():
    ids = np.array([[0, 5], [2, 0], [-1, 1]], np.int32)
    _check(ids, 3, 2)
