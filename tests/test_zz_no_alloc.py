"""qmoe_forward_noalloc: the forward for callers that cannot allocate device
memory at call time (an engine plugin with a fixed memory plan and no scratch
buffer, a serving loop that must stay out of the allocator).  It must give the
regular entry point's result, call after call, from the library's built-in
scratch array, and refuse work that needs more scratch than that array holds.
This file is collected last so that a failure here cannot hide another test.
"""
import ctypes

import numpy as np
import pytest
import torch

import weight_only_quantized_moe_gb300 as q
from synth import Workload, make_inputs, make_layer
from tests.gpu_util import assert_parity, device_inputs, device_layer, ensure_built, run_forward

pytestmark = pytest.mark.gpu


def _call_noalloc(dl, x, ids, w, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return q.lib().qmoe_forward_noalloc(ctypes.byref(dl.struct), ctypes.c_void_p(x.data_ptr()), x.shape[0],
                                        ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                        ids.shape[1], ctypes.c_void_p(out.data_ptr()), stream)


@pytest.mark.parametrize("qt,act", [("int4", "bf16"), ("int8", "f16")])
def test_noalloc_matches_regular_forward_on_consecutive_calls(qt, act):
    ensure_built()
    wl = Workload("noalloc", 8, 2, 384, 256, qt, 128 if qt == "int4" else -1, act, False, 0.0, (1,))
    dl = device_layer(make_layer(wl, seed=4))
    inp = make_inputs(wl, 40, seed=5)
    x, ids, w = device_inputs(wl, inp)
    want, _ = run_forward(dl, x, ids, w)
    want = want.double().cpu().numpy()
    for _ in range(2):
        out = torch.full_like(x, float("nan"))
        assert _call_noalloc(dl, x, ids, w, out) == q.QMOE_OK
        torch.cuda.synchronize()
        assert_parity(out.double().cpu().numpy(), want, "noalloc vs qmoe_forward")


def test_noalloc_rejects_work_beyond_its_scratch():
    ensure_built()
    wl = Workload("noalloc_big", 8, 2, 4096, 4096, "int4", 128, "f16", False, 0.0, (1,))
    dl = device_layer(make_layer(wl, seed=1))
    M = 4096  # needs far more than the built-in 64 MiB scratch
    assert q.qmoe_workspace_size(dl, M, 2) > (64 << 20)
    x = torch.zeros((M, wl.H), dtype=torch.float16, device="cuda")
    ids = torch.zeros((M, 2), dtype=torch.int32, device="cuda")
    w = torch.zeros((M, 2), dtype=torch.float32, device="cuda")
    out = torch.empty_like(x)
    assert _call_noalloc(dl, x, ids, w, out) == q.QMOE_ERR_WORKSPACE
