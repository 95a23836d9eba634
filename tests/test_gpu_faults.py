"""Device-side failure path: a pipeline wait that can never complete must give
up within its time limit, report QMOE_ERR_TIMEOUT through the workspace status
word and leave the CUDA context usable (no trap, no hang)."""
import time

import pytest

import oracle
import weight_only_quantized_moe_gb300 as q
from synth import Workload, make_inputs, make_layer
from tests.gpu_util import assert_parity, device_inputs, device_layer, ensure_built, run_forward

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pair", [0, 1])
def test_withheld_stage_times_out_and_context_survives(pair):
    """Single CTAs, and CTA pairs (CTA 0 withholds its stage; its peer's waits on
    the pair's MMAs then run out as well)."""
    ensure_built()
    wl = Workload("fault", 8, 2, 256, 256, "int4", 128, "f16", False, 0.0, (1,))
    L = make_layer(wl, seed=1)
    dl = device_layer(L)
    inp = make_inputs(wl, 12, seed=2)
    x, ids, w = device_inputs(wl, inp)
    t0 = time.time()
    _, st = run_forward(dl, x, ids, w, opts=q.make_options(fault_injection=1, cta_pair=pair), check_status=False)
    elapsed = time.time() - t0
    assert st == q.QMOE_ERR_TIMEOUT, q.status_string(st)
    assert elapsed < 30
    # the context is intact: a normal forward right after is correct
    out, st = run_forward(dl, x, ids, w)
    assert st == q.QMOE_OK
    ref = oracle.moe_forward(L, inp.x, inp.topk_ids, inp.topk_weights)
    assert_parity(out.float().cpu().numpy(), ref, "after timeout")
