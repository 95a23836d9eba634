"""qmoe_forward_noalloc: the forward for callers that cannot allocate device
memory at call time (an engine plugin with a fixed memory plan and no scratch
buffer, a serving loop that must stay out of the allocator).  It must give the
regular entry point's result bit for bit, call after call, from the library's
built-in scratch array, report device-side faults through
qmoe_read_noalloc_status, and refuse work that needs more scratch than that
array holds.  This file is collected last so that a failure here cannot hide
another test.
"""
import ctypes

import numpy as np
import pytest
import torch

import weight_only_quantized_moe_gb300 as q
from synth import Workload, make_inputs, make_layer
from tests.gpu_util import device_inputs, device_layer, ensure_built, run_forward

pytestmark = pytest.mark.gpu


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _call_noalloc(dl, x, ids, w, out):
    return q.lib().qmoe_forward_noalloc(ctypes.byref(dl.struct), ctypes.c_void_p(x.data_ptr()), x.shape[0],
                                        ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                        ids.shape[1], ctypes.c_void_p(out.data_ptr()), _stream())


def _read_status():
    return q.lib().qmoe_read_noalloc_status(_stream())


@pytest.mark.parametrize("qt,act", [("int4", "bf16"), ("int8", "f16")])
def test_noalloc_matches_regular_forward_on_consecutive_calls(qt, act):
    """Both entry points run the same kernels with the same plan and a fixed-order
    reduction, so the outputs agree bit for bit.  A call with another M in
    between leaves other contents (status word, padding rows, chunk table) in
    the shared scratch; the next call must not depend on them."""
    ensure_built()
    wl = Workload("noalloc", 8, 2, 384, 256, qt, 128 if qt == "int4" else -1, act, False, 0.0, (1,))
    dl = device_layer(make_layer(wl, seed=4))
    inp = make_inputs(wl, 40, seed=5)
    x, ids, w = device_inputs(wl, inp)
    want, _ = run_forward(dl, x, ids, w)
    other = make_inputs(wl, 97, seed=6)
    xo, ido, wo = device_inputs(wl, other)
    want_o, _ = run_forward(dl, xo, ido, wo)
    for rep in range(2):
        out = torch.full_like(x, float("nan"))
        assert _call_noalloc(dl, x, ids, w, out) == q.QMOE_OK
        assert _read_status() == q.QMOE_OK
        assert torch.equal(out, want), f"call {rep}: noalloc output differs from qmoe_forward"
        out_o = torch.full_like(xo, float("nan"))
        assert _call_noalloc(dl, xo, ido, wo, out_o) == q.QMOE_OK
        assert _read_status() == q.QMOE_OK
        assert torch.equal(out_o, want_o), f"call {rep}: noalloc output (M=97) differs from qmoe_forward"


def test_noalloc_reports_device_faults_through_its_status():
    """A top-k id outside [0, E) is only seen on the device; the status accessor
    reads it from the shared scratch, and the next good call clears it."""
    ensure_built()
    wl = Workload("noalloc_bad", 8, 2, 384, 256, "int4", 128, "f16", False, 0.0, (1,))
    dl = device_layer(make_layer(wl, seed=2))
    inp = make_inputs(wl, 16, seed=3)
    x, ids, w = device_inputs(wl, inp)
    bad = ids.clone()
    bad[3, 1] = wl.E
    out = torch.empty_like(x)
    assert _call_noalloc(dl, x, bad, w, out) == q.QMOE_OK
    assert _read_status() == q.QMOE_ERR_BAD_EXPERT_ID
    assert _call_noalloc(dl, x, ids, w, out) == q.QMOE_OK
    assert _read_status() == q.QMOE_OK
    want, _ = run_forward(dl, x, ids, w)
    assert torch.equal(out, want)


def test_noalloc_rejects_work_beyond_its_scratch():
    ensure_built()
    wl = Workload("noalloc_big", 8, 2, 4096, 4096, "int4", 128, "f16", False, 0.0, (1,))
    dl = device_layer(make_layer(wl, seed=1))
    M = 4096  # needs far more than the built-in 64 MiB scratch
    assert q.qmoe_workspace_size(dl, M, 2) > (64 << 20)
    x = torch.zeros((M, wl.H), dtype=torch.float16, device="cuda")
    ids = torch.zeros((M, 2), dtype=torch.int32, device="cuda")
    w = torch.zeros((M, 2), dtype=torch.float32, device="cuda")
    out = torch.full_like(x, 1.0)
    assert _call_noalloc(dl, x, ids, w, out) == q.QMOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool(torch.all(out == 1.0)), "a rejected call must launch nothing"
    assert np.isfinite(float(out[0, 0]))
