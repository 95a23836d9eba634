"""The dense linear layer on the GPU (qmoe_linear_forward, through the C ABI)
against the float64 oracle: every weight format ("Add GPTQ Marlin 2:4 sparse
structured support": 4 or 8 bits, group 128 or channel-wise, dense or 2:4
sparse; plus act-order and zero points), batch sizes that span one and several
token chunks and a ragged tail, forced split-K and token tiles, and a
Mixtral-sized matrix."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_moe_gb300 as q
from synth import make_linear, make_linear_inputs
from tests.gpu_util import assert_parity, ensure_built

pytestmark = pytest.mark.gpu

_TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}

FORMATS = [("int4", 128, "f16", False), ("int4", 128, "bf16", True), ("int4", -1, "bf16", False),
           ("int4zp", 128, "bf16", True), ("int4zp", -1, "f16", False), ("int4s24", 128, "f16", False),
           ("int4s24", -1, "bf16", False), ("int8", -1, "bf16", False), ("int8", -1, "f16", False),
           ("int8g", 128, "f16", False), ("int8s24", -1, "bf16", False), ("int8s24", 128, "f16", False),
           ("int8s24", 128, "bf16", False)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


_CACHE = {}


def _layer(qt, gs, act, ao, N=384, K=512):
    key = (qt, gs, act, ao, N, K)
    if key not in _CACHE:
        lin = make_linear(N, K, qt, gs, act, act_order=ao, seed=5)
        dl = q.DeviceLinear.from_canonical(qt, act, lin.q, lin.s, gs, lin.z, lin.g_idx)
        _CACHE[key] = (lin, dl, oracle.dequant_linear(lin))
    return _CACHE[key]


def _run(dl, x, opts=None):
    ws = q.alloc_workspace(q.qmoe_linear_workspace_size(dl, x.shape[0], opts), x.device)
    ws.fill_(0xFF)  # NaN in every float type: an unwritten workspace byte read back would show
    out = torch.full((x.shape[0], dl.N), float("nan"), dtype=x.dtype, device=x.device)
    q.qmoe_linear_forward(dl, x, out=out, workspace=ws, opts=opts)
    assert q.qmoe_read_device_status(ws) == q.QMOE_OK
    return out.double().cpu().numpy()


@pytest.mark.parametrize("qt,gs,act,ao", FORMATS)
@pytest.mark.parametrize("M", [1, 16, 37, 200])
def test_linear_parity(qt, gs, act, ao, M):
    lin, dl, W = _layer(qt, gs, act, ao)
    xs = make_linear_inputs(lin.q.shape[1], M, act, seed=M)
    got = _run(dl, torch.from_numpy(xs).to(_TORCH[act]).cuda())
    assert_parity(got, oracle.linear_forward(xs, W), f"linear {qt} g{gs} {act} ao={ao} M={M}")


@pytest.mark.parametrize("qt,gs,act,ao", [FORMATS[0], FORMATS[1], FORMATS[5], FORMATS[10], FORMATS[11]])
@pytest.mark.parametrize("split1,tile", [(2, 0), (4, 16), (1, 32), (3, 128)])
def test_linear_forced_split_and_tile(qt, gs, act, ao, split1, tile):
    lin, dl, W = _layer(qt, gs, act, ao)
    M = 45
    xs = make_linear_inputs(lin.q.shape[1], M, act, seed=3)
    got = _run(dl, torch.from_numpy(xs).to(_TORCH[act]).cuda(), q.make_options(split1, 0, tile))
    assert_parity(got, oracle.linear_forward(xs, W), f"linear {qt} split {split1} tile {tile}")


@pytest.mark.parametrize("qt,gs,act", [("int4", 128, "f16"), ("int4s24", 128, "f16"), ("int8s24", -1, "bf16")])
@pytest.mark.parametrize("M", [1, 16, 256])
def test_linear_mixtral_sized(qt, gs, act, M):
    """A 14336 x 4096 weight (the Mixtral-8x7B expert's gate projection shape) at
    the default plan, every output element checked."""
    lin, dl, W = _layer(qt, gs, act, False, N=14336, K=4096)
    xs = make_linear_inputs(4096, M, act, seed=M + 1)
    got = _run(dl, torch.from_numpy(xs).to(_TORCH[act]).cuda())
    assert_parity(got, oracle.linear_forward(xs, W), f"linear 14336x4096 {qt} M={M}")


def test_linear_deterministic_and_m_zero():
    lin, dl, W = _layer("int4", 128, "bf16", True)
    xs = make_linear_inputs(512, 33, "bf16", seed=8)
    x = torch.from_numpy(xs).to(torch.bfloat16).cuda()
    a = _run(dl, x)
    b = _run(dl, x)
    assert np.array_equal(a, b)
    empty = torch.empty((0, 512), dtype=torch.bfloat16, device="cuda")
    out = q.qmoe_linear_forward(dl, empty, workspace=q.alloc_workspace(256))
    assert out.shape == (0, 384)
