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


def _al256(n):
    return (n + 255) // 256 * 256


@pytest.mark.parametrize("M,k,E,zipf", [(1, 2, 8, 0.0), (5, 2, 8, 0.0), (16, 6, 160, 1.1), (300, 2, 8, 0.0),
                                        (512, 2, 8, 0.0), (170, 6, 160, 1.1), (513, 2, 8, 0.0), (1024, 6, 160, 1.1)])
def test_forward_grouping_matches_oracle(M, k, E, zipf):
    """The grouping a forward computes (by the fused align+gather kernel for up to
    1024 pairs, by moe_align above) is bit-exact: it is read back from the
    workspace, whose first regions are the status word (256 bytes), sorted_ids
    [cap] and expert_ids [cap / 16], each rounded up to 256 bytes, then the padded
    total; cap = P + 15 E rounded up to 16."""
    import torch
    import oracle
    import weight_only_quantized_moe_gb300 as q
    from synth import Workload, make_inputs, make_layer
    from tests.gpu_util import device_inputs, device_layer
    wl = Workload("grp", E, k, 128, 128, "int4", 128, "f16", False, zipf, (1,))
    dl = device_layer(make_layer(wl, seed=1))
    inp = make_inputs(wl, M, seed=M)
    x, ids, w = device_inputs(wl, inp)
    ws = q.alloc_workspace(q.qmoe_workspace_size(dl, M, k))
    ws.fill_(0x7F)
    q.qmoe_forward(dl, x, ids, w, workspace=ws)
    torch.cuda.synchronize()
    P = M * k
    cap = (P + E * 15 + 15) // 16 * 16
    nblocks = (cap + 15) // 16
    want_sorted, want_expert, want_total = oracle.moe_align(inp.topk_ids, E, 16, cap)
    raw = ws.cpu().numpy()
    got_sorted = raw[256:256 + 4 * cap].view(np.int32)
    off_e = 256 + _al256(4 * cap)
    got_expert = raw[off_e:off_e + 4 * nblocks].view(np.int32)
    off_s = off_e + _al256(4 * nblocks)
    got_total = int(raw[off_s:off_s + 4].view(np.int32)[0])
    assert got_total == want_total
    np.testing.assert_array_equal(got_sorted, want_sorted)
    np.testing.assert_array_equal(got_expert, want_expert[:nblocks])
    assert q.qmoe_read_device_status(ws) == q.QMOE_OK
