"""Helpers shared by the GPU tests: upload synthetic layers, run the CUDA path
through the C ABI, and measure parity against the oracle."""
import numpy as np
import torch

import weight_only_quantized_moe_gb300 as q
from weight_only_quantized_moe_gb300 import build as _build

# Parity bar for layer outputs (relative to the oracle's float64 result):
# max |err| <= 2e-2 * rms(ref) and ||err||_2 <= 5e-3 * ||ref||_2.
MAX_ERR_REL_RMS = 2e-2
REL_L2 = 5e-3

_TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}


def ensure_built():
    _build.build()
    q.lib()


def device_layer(layer, device="cuda"):
    wl = layer.wl
    return q.DeviceLayer.from_canonical(wl.qt, wl.act, layer.q13, layer.s13, layer.q2, layer.s2,
                                        layer.g13, layer.g2, device=device, z13=layer.z13, z2=layer.z2,
                                        group_size=wl.group_size)


def device_inputs(wl, inp, device="cuda"):
    x = torch.from_numpy(inp.x).to(_TORCH[wl.act]).to(device)
    ids = torch.from_numpy(np.ascontiguousarray(inp.topk_ids, np.int32)).to(device)
    w = torch.from_numpy(np.ascontiguousarray(inp.topk_weights, np.float32)).to(device)
    return x, ids, w


def run_forward(dl, x, ids, w, opts=None, check_status=True, ws_fill=0xFF):
    ws = q.alloc_workspace(q.qmoe_workspace_size(dl, x.shape[0], ids.shape[1], opts), x.device)
    if ws_fill is not None:
        # all-ones bytes are NaN in every float type: a read of a workspace byte the
        # forward did not write first would show up in the output
        ws.fill_(ws_fill)
    out = q.qmoe_forward(dl, x, ids, w, workspace=ws, opts=opts)
    st = q.qmoe_read_device_status(ws)
    if check_status:
        assert st == q.QMOE_OK, q.status_string(st)
    return out, st


def parity(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = got - ref
    rms = float(np.sqrt(np.mean(ref * ref)))
    max_rel = float(np.max(np.abs(err)) / rms) if rms > 0 else float(np.max(np.abs(err)))
    rel_l2 = float(np.linalg.norm(err) / np.linalg.norm(ref)) if rms > 0 else 0.0
    return max_rel, rel_l2


def assert_parity(got, ref, what=""):
    max_rel, rel_l2 = parity(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert max_rel <= MAX_ERR_REL_RMS and rel_l2 <= REL_L2, f"{what}: max|err|/rms={max_rel:.3e} relL2={rel_l2:.3e}"
    return max_rel, rel_l2
