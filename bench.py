#!/usr/bin/env python
"""Benchmark of the fused weight-only-quantized MoE layer on GB300.

One step = one full layer forward (moe_align, token gather, gate/up GEMM with
fused SiLU*up, down GEMM with the routing weight, top-k reduce) over one batch
of M tokens of a synthetic workload shaped like the pages' models.  Prints ONE
JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--M M] [--no-sweep] [--workloads A,B]

The headline (value, e2e, roofline, clocks) is --workload at --M over exactly K
timed steps.  The same line's "workloads" list then reports every workload at
every batch size it is measured at (Mixtral-8x7B int4 decode, act-order, int8,
the DeepSeek-V2-like layer, Mixtral-8x22B prefill, 2:4-sparse int4), each over
at least K steps and at least 0.3 s of timed work, with its own per-kernel
times, roofline and clock record.

--impl reference times the CPU oracle (float64 numpy) on a bounded sample of
the same workload; it is the only other place this file runs the oracle.
Multi-GPU (torchrun): every rank runs the same workload on its own GPU
(independent replicas; the layer is not sharded), value = all ranks' tokens /
max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import WORKLOADS, make_inputs, make_layer  # noqa: E402

METRIC = "quant-MoE layer tokens/s, TFLOP/s & weight GB/s vs roofline, M=1..8192"
DEFAULT_WORKLOAD = "mixtral8x7b_w4"
DEFAULT_M = 16
L2_BYTES = 129 * 1024 * 1024
LAUNCH_NAMES = ["moe_align", "gather", "gemm_gate_up", "silu_reduce", "inter_rescale", "gemm_down", "out_reduce"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--M", type=int, default=None)
    ap.add_argument("--no-sweep", action="store_true", help="headline workload only")
    ap.add_argument("--workloads", type=lambda v: v.split(","), default=None,
                    help="comma-separated subset of the reported workloads")
    ap.add_argument("--cpu-sample-s", type=float, default=20.0)
    ap.add_argument("--ncu-pass", action="store_true",
                    help="no timing: run each reported (workload, M) forward 3 times on one weight copy, for an "
                         "ncu capture of per-launch counters (the 3rd forward of each entry is the one to read)")
    ap.add_argument("--record-traffic", nargs=2, metavar=("NCU_CSV", "NCU_PASS_LOG"), default=None,
                    help="no GPU: write profiles/dram_traffic.txt from an ncu --csv capture of --ncu-pass "
                         "(dram__bytes_read.sum, dram__bytes_write.sum, gpu__time_duration.sum) and that run's stdout")
    return ap.parse_args()


def peaks():
    """HBM copy bandwidth (GB/s) and dense bf16 tensor rate (TFLOP/s, burst and
    sustained) measured on this GPU pool, else the recipe's fallback figures."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm": float(d["hbm_gbs"]), "tc_burst": float(d["bf16_tflops"]),
                "tc_sust": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "src": "measured"}
    return {"hbm": 6800.0, "tc_burst": 1900.0, "tc_sust": 1700.0, "src": "fallback"}


def workload_config(wl, M, extra=None):
    cfg = {"workload": f"{wl.name}: E={wl.E} top-{wl.k} H={wl.H} I={wl.I} {wl.qt}"
                       f"{' g128' if wl.group_size == 128 else ' per-column'}"
                       f"{' 2:4-sparse' if wl.qt == 'int4s24' else ''}{' act-order' if wl.act_order else ''}"
                       f" {wl.act} activations, M={M}",
           "E": wl.E, "top_k": wl.k, "hidden": wl.H, "intermediate": wl.I, "quant": wl.qt,
           "group_size": wl.group_size, "act_order": wl.act_order, "act_dtype": wl.act, "M": M}
    if extra:
        cfg.update(extra)
    return cfg


# ----------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ----------------------------------------------------------------------------
def oracle_sample(wl, layer, inp, budget_s):
    """Time the oracle on the first tokens of the batch, one token at a time,
    until about budget_s seconds of CPU work; returns (tokens, seconds)."""
    import oracle
    t0 = time.perf_counter()
    n = 0
    M = inp.x.shape[0]
    while n < M:
        oracle.moe_forward_rows(layer, inp.x, inp.topk_ids, inp.topk_weights, [n])
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return n, time.perf_counter() - t0


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """Slowest rank's time: every rank contributes its own ms, all get the max."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(tokens_per_rank: int, world: int, ms: float) -> float:
    """Replicas: every rank processes its own batch; value = all ranks' tokens / slowest rank's time."""
    return world * tokens_per_rank / (ms * 1e-3)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    """Samples the SM clock and the clock-event reasons of one GPU every ~0.5 ms
    while the timed region runs (NVML through ctypes; read-only queries)."""
    SM = 1  # NVML_CLOCK_SM
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index):
        self.dev = device_index
        self.rows = []
        self.max_mhz = None
        self.err = None
        self.nvml = None
        self.handle = None
        self.thread = None
        self.stop = None

    def _open(self):
        import ctypes
        import torch
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        h = ctypes.c_void_p()
        uuid = "GPU-" + str(torch.cuda.get_device_properties(self.dev).uuid)
        if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByUUID failed")
        self.nvml, self.handle = nv, h
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, self.SM, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn if fn is not None else nv.nvmlDeviceGetCurrentClocksThrottleReasons

    def _loop(self):
        import ctypes
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        while not self.stop.is_set():
            if (self.nvml.nvmlDeviceGetClockInfo(self.handle, self.SM, ctypes.byref(c)) == 0 and
                    self.reasons_fn(self.handle, ctypes.byref(r)) == 0):
                self.rows.append((float(c.value), int(r.value)))
            time.sleep(0.0005)

    def __enter__(self):
        import threading
        try:
            self._open()
            self.stop = threading.Event()
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.rows and time.time() - t0 < 2.0:  # first sample before the timed region
                time.sleep(0.001)
        except Exception as e:  # no NVML on this host
            self.err = f"nvml unavailable: {e}"
        return self

    def __exit__(self, *a):
        if self.thread is not None:
            self.stop.set()
            self.thread.join(timeout=2.0)

    def summary(self):
        if self.err is not None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [self.err], "samples": 0}
        rows = self.rows[1:] if len(self.rows) > 1 else self.rows  # the first sample precedes the region
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"], "samples": 0}
        reasons = sorted({name for _, bits in rows for b, name in self.REASONS.items() if bits & b})
        return {"sm_mhz": statistics.median(c for c, _ in rows), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# work per call and rooflines (host arithmetic)
# ----------------------------------------------------------------------------
def algorithmic_bytes(wl, expert_w13_bytes, expert_w2_bytes, topk_ids, M):
    """Bytes the method must move per layer call: the touched experts' packed
    weights and scales, x in, intermediate write + read, out.  Per GEMM launch:
    gate/up = touched W13 + gathered tokens read + intermediate written;
    down = touched W2 + intermediate read + per-pair fp32 outputs written."""
    d = int(len(np.unique(topk_ids)))
    P = M * wl.k
    act = 2
    gemm1 = d * expert_w13_bytes + P * wl.H * act + P * wl.I * act
    gemm2 = d * expert_w2_bytes + P * wl.I * act + P * wl.H * 4
    total = d * (expert_w13_bytes + expert_w2_bytes) + M * wl.H * act * 2 + 2 * P * wl.I * act
    return {"distinct_experts": d, "gemm_gate_up": gemm1, "gemm_down": gemm2, "layer": total,
            "weights": d * (expert_w13_bytes + expert_w2_bytes)}


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "weight_only_quantized_moe_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, M, kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu record, or None
    if there is none for this workload or the kernel source changed since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    cur = kernel_source_hash()
    with open(path) as f:
        for line in f:
            p = line.split()
            if len(p) >= 5 and not p[0].startswith("#") and p[0] == workload and int(p[1]) == M and p[2] == kernel:
                return int(p[3]) if p[4] == cur else None
    return None


def gemm_flops(wl, M, kernel):
    P = M * wl.k
    return 2.0 * P * (2 * wl.I if kernel == "gemm_gate_up" else wl.I) * wl.H


def roofline_entry(wl, M, ms, kernel_ms, by, pk):
    """Roofline of one (workload, M): the dominant GEMM launch against its binding
    peak (HBM or tensor, by its arithmetic intensity against the peaks' ratio),
    and the whole layer against both peaks."""
    hbm, tc_burst, tc_sust = pk["hbm"], pk["tc_burst"], pk["tc_sust"]
    dominant = max(("gemm_gate_up", "gemm_down"), key=lambda n: kernel_ms[n])
    kflops = gemm_flops(wl, M, dominant)
    ks = kernel_ms[dominant] * 1e-3
    if kflops / by[dominant] > tc_burst * 1e12 / (hbm * 1e9):
        ach = kflops / ks / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": tc_burst, "unit": "TFLOP/s", "frac": ach / tc_burst,
                "frac_of_sustained_peak": ach / tc_sust,
                "peak_source": f"{pk['src']} bf16_tflops burst (cuBLAS bf16 GEMM; the f16 MMAs run at the bf16 rate)",
                "algorithmic_flops_per_launch": kflops}
    else:
        ach = by[dominant] / ks / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "peak_source": f"{pk['src']} hbm_gbs (copy bandwidth)",
                "algorithmic_bytes_per_launch": by[dominant]}
    roof["kernel"] = dominant
    roof["kernel_ms"] = kernel_ms[dominant]
    t = ms * 1e-3
    flops = wl.flops(M)
    layer = {"tokens_per_s": M / t, "tflops": flops / t / 1e12, "weight_gbs": by["weights"] / t / 1e9,
             "frac_hbm_weights": by["weights"] / t / 1e9 / hbm, "frac_hbm_layer": by["layer"] / t / 1e9 / hbm,
             "frac_tensor_layer": flops / t / 1e12 / tc_burst,
             "binding": "tensor" if flops / by["layer"] > tc_burst * 1e12 / (hbm * 1e9) else "hbm"}
    layer["frac_binding"] = layer["frac_tensor_layer"] if layer["binding"] == "tensor" else layer["frac_hbm_layer"]
    return roof, layer


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
# every (workload, M) the layer is reported at, besides the headline
REPORTED = (("mixtral8x7b_w4", (1, 4, 8, 16, 64)), ("mixtral8x7b_w4_actorder", (1, 16, 128, 512)),
            ("mixtral8x7b_w8", (1, 16, 128, 512)), ("deepseekv2_w8", (1, 32, 256, 1024)),
            ("mixtral8x22b_w4", (2048, 4096, 8192)), ("mixtral8x7b_w4s24", (1, 16, 64)),
            ("mixtral8x7b_w8s24", (1, 16, 64)))
MIN_TIMED_S = 0.3      # timed region per reported entry (clock samples every ~0.5 ms)
MAX_ROTATION_BYTES = 24 << 30
# dense linear layer (one weight matrix, no routing): dense and 2:4-sparse, 4 and 8 bits
LINEAR_REPORTED = (("int4", 128, "f16"), ("int4s24", 128, "f16"), ("int8", -1, "bf16"), ("int8s24", -1, "bf16"))
LINEAR_SHAPE = (28672, 4096)   # N output features, K input features (a Mixtral-8x7B expert's gate+up)
LINEAR_MS = (1, 16, 128)


class GpuWorkload:
    """One workload's packed layer on the device, rotated across copies so that
    no step finds its experts' weights in L2."""

    def __init__(self, q, wl, dev):
        import torch
        self.q, self.wl, self.dev = q, wl, dev
        layer = make_layer(wl, seed=0)
        self.base = q.DeviceLayer.from_canonical(wl.qt, wl.act, layer.q13, layer.s13, layer.q2, layer.s2, layer.g13,
                                                 layer.g2, device=dev, z13=layer.z13, z2=layer.z2,
                                                 group_size=wl.group_size)
        del layer
        b = self.base
        fs = b.s13 is not None  # float32 scales per output feature, outside the packed blocks
        self.w13_e = b.w13.numel() // wl.E + (2 * wl.I * 4 if fs else 0)
        self.w2_e = b.w2.numel() // wl.E + (wl.H * 4 if fs else 0)
        self.copies = [b]
        self.torch = torch

    def ensure_copies(self, touched_bytes):
        """Enough copies that one lap of the rotation touches 3x the L2 size."""
        b = self.base
        want = min(16, math.ceil(3 * L2_BYTES / max(1, touched_bytes)) + 1)
        want = max(1, min(want, MAX_ROTATION_BYTES // max(1, b.weight_bytes())))
        while len(self.copies) < want:
            c = lambda t: None if t is None else t.clone()
            self.copies.append(self.q.DeviceLayer(b.qt, b.E, b.H, b.I, b.act, b.w13.clone(), b.w2.clone(), c(b.s13),
                                                  c(b.s2), c(b.perm13), b.group_size))
        return len(self.copies)

    def inputs(self, M):
        torch = self.torch
        inp = make_inputs(self.wl, M, seed=0)
        x = torch.from_numpy(inp.x).to(self.base.torch_dtype).to(self.dev)
        ids = torch.from_numpy(inp.topk_ids).to(self.dev)
        w = torch.from_numpy(inp.topk_weights).to(self.dev)
        return inp, x, ids, w

    def measure(self, M, steps, warmup, world=1, min_s=0.0):
        """Time `steps` forwards (more when min_s asks for a longer timed region),
        then the same number again with CUDA events around each kernel launch."""
        torch, q, wl = self.torch, self.q, self.wl
        inp, x, ids, w = self.inputs(M)
        by = algorithmic_bytes(wl, self.w13_e, self.w2_e, inp.topk_ids, M)
        ncop = self.ensure_copies(by["weights"])
        out = torch.empty_like(x)
        ws = q.alloc_workspace(q.qmoe_workspace_size(self.base, M, wl.k), self.dev)
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(warmup):
            q.qmoe_forward(self.copies[i % ncop], x, ids, w, out=out, workspace=ws)
        e1.record(stream)
        torch.cuda.synchronize()
        st = q.qmoe_read_device_status(ws)
        if st != q.QMOE_OK:
            raise RuntimeError(f"{wl.name} M={M}: device status after warm-up: {q.status_string(st)}")
        if min_s > 0 and warmup > 0:
            est = e0.elapsed_time(e1) / warmup * 1e-3
            steps = int(min(4000, max(steps, math.ceil(min_s / max(est, 1e-6)))))
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        with ClockSampler(self.dev.index) as clk:
            e0.record(stream)
            for i in range(steps):
                q.qmoe_forward(self.copies[i % ncop], x, ids, w, out=out, workspace=ws)
            e1.record(stream)
            torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        # second pass: CUDA events on the launch stream around each kernel launch
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(LAUNCH_NAMES))] for _ in range(steps)]
        launches = 0
        for i in range(steps):
            launches += q.qmoe_forward_profiled(self.copies[i % ncop], x, ids, w, out, ws, evs[i])
        torch.cuda.synchronize()
        kms = {name: sum(evs[i][2 * j].elapsed_time(evs[i][2 * j + 1]) for i in range(steps)) / steps
               for j, name in enumerate(LAUNCH_NAMES)}
        st = q.qmoe_read_device_status(ws)
        if st != q.QMOE_OK:
            raise RuntimeError(f"{wl.name} M={M}: device status: {q.status_string(st)}")
        return {"M": M, "ms": ms, "steps": steps, "clocks": clk.summary(), "inp": inp, "kernel_ms": kms,
                "launches_per_step": launches / steps, "bytes": by, "copies": ncop, "x": x, "ids": ids, "w": w}

    def release(self):
        self.copies = []
        self.base = None
        self.torch.cuda.empty_cache()


class GpuLinear:
    """A dense linear layer's packed weight on the device, rotated across copies."""

    def __init__(self, q, qt, gs, act, N, K, dev):
        import torch
        from synth import make_linear
        self.q, self.qt, self.gs, self.act, self.N, self.K, self.dev, self.torch = q, qt, gs, act, N, K, dev, torch
        lin = make_linear(N, K, qt, gs, act, seed=0)
        self.base = q.DeviceLinear.from_canonical(qt, act, lin.q, lin.s, gs, lin.z, lin.g_idx, device=dev)
        del lin
        b = self.base
        self.wbytes = b.w.numel() + (4 * b.s.numel() if b.s is not None else 0)
        n = max(1, min(16, math.ceil(3 * L2_BYTES / self.wbytes) + 1))
        self.copies = [b] + [q.DeviceLinear(qt, N, K, act, b.w.clone(), None if b.s is None else b.s.clone(), None, gs)
                             for _ in range(n - 1)]

    def measure(self, M, steps, warmup, min_s=0.0):
        torch, q = self.torch, self.q
        from synth import make_linear_inputs
        x = torch.from_numpy(make_linear_inputs(self.K, M, self.act, seed=0)).to(self.base.torch_dtype).to(self.dev)
        out = torch.empty((M, self.N), dtype=x.dtype, device=self.dev)
        ws = q.alloc_workspace(q.qmoe_linear_workspace_size(self.base, M), self.dev)
        nc = len(self.copies)
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(warmup):
            q.qmoe_linear_forward(self.copies[i % nc], x, out=out, workspace=ws)
        e1.record(stream)
        torch.cuda.synchronize()
        if q.qmoe_read_device_status(ws) != q.QMOE_OK:
            raise RuntimeError(f"linear {self.qt} M={M}: device status after warm-up")
        if min_s > 0 and warmup > 0:
            est = e0.elapsed_time(e1) / warmup * 1e-3
            steps = int(min(4000, max(steps, math.ceil(min_s / max(est, 1e-6)))))
        with ClockSampler(self.dev.index) as clk:
            e0.record(stream)
            for i in range(steps):
                q.qmoe_linear_forward(self.copies[i % nc], x, out=out, workspace=ws)
            e1.record(stream)
            torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        plan = q.qmoe_linear_describe_plan(self.base, M)
        return {"ms": ms, "steps": steps, "clocks": clk.summary(), "plan": plan}

    def entry(self, M, r, pk):
        t = r["ms"] * 1e-3
        byts = self.wbytes + M * self.K * 2 + M * self.N * 2
        flops = 2.0 * M * self.N * self.K
        hbm_frac = byts / t / 1e9 / pk["hbm"]
        tc_frac = flops / t / 1e12 / pk["tc_burst"]
        bound = "tensor" if flops / byts > pk["tc_burst"] * 1e12 / (pk["hbm"] * 1e9) else "hbm"
        return {"layer": "dense linear", "quant": self.qt, "group_size": self.gs, "act_dtype": self.act,
                "N": self.N, "K": self.K, "M": M, "ms": r["ms"], "steps": r["steps"],
                "weight_bytes": self.wbytes, "weight_gbs": self.wbytes / t / 1e9, "tflops": flops / t / 1e12,
                "frac_hbm": hbm_frac, "frac_tensor": tc_frac, "binding": bound,
                "frac_binding": tc_frac if bound == "tensor" else hbm_frac,
                "plan": {k: r["plan"][k] for k in ("token_tile", "issuers", "split1")}, "clocks": r["clocks"],
                "rotation_copies": len(self.copies)}

    def release(self):
        self.copies = []
        self.base = None
        self.torch.cuda.empty_cache()


def e2e_host(gw, r, steps, warmup, world):
    """The same layer end to end through the host-buffer entry point: every step
    copies x, the top-k ids and weights from pinned host memory to the device,
    runs the forward, and copies out back."""
    torch, q, wl = gw.torch, gw.q, gw.wl
    M = r["M"]
    xh = r["x"].cpu().pin_memory()
    idh = r["ids"].cpu().pin_memory()
    wh = r["w"].cpu().pin_memory()
    outh = torch.empty_like(xh).pin_memory()
    wsh = q.alloc_workspace(q.qmoe_workspace_size_host(gw.base, M, wl.k), gw.dev)
    ncop = len(gw.copies)
    for i in range(warmup):
        q.qmoe_forward_host(gw.copies[i % ncop], xh, idh, wh, outh, wsh)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        q.qmoe_forward_host(gw.copies[i % ncop], xh, idh, wh, outh, wsh)
    e1.record(stream)
    torch.cuda.synchronize()
    return max_over_ranks(e0.elapsed_time(e1) / steps, world, gw.dev)


def entry_line(wl, r, pk):
    roof, layer = roofline_entry(wl, r["M"], r["ms"], r["kernel_ms"], r["bytes"], pk)
    roof["traffic"] = recorded_traffic(wl.name, r["M"], roof["kernel"])
    return {"workload": wl.name, "M": r["M"], "ms": r["ms"], "steps": r["steps"], **layer,
            "distinct_experts": r["bytes"]["distinct_experts"], "roofline": roof,
            "kernel_ms": {n: round(v, 5) for n, v in r["kernel_ms"].items()}, "clocks": r["clocks"],
            "rotation_copies": r["copies"]}


def run_gpu(args, rank, world):
    import torch

    import weight_only_quantized_moe_gb300 as q
    from weight_only_quantized_moe_gb300 import build as qbuild

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    qbuild.build()
    q.lib()
    pk = peaks()
    wl = WORKLOADS[args.workload]
    M = args.M or (DEFAULT_M if DEFAULT_M in wl.Ms else wl.Ms[0])
    gw = GpuWorkload(q, wl, dev)
    main = gw.measure(M, args.steps, args.warmup, world)
    ms = max_over_ranks(main["ms"], world, dev)
    e2e_ms = e2e_host(gw, main, args.steps, args.warmup, world)
    entries = []
    if not args.no_sweep:
        todo = [(n, Ms) for n, Ms in REPORTED if args.workloads is None or n in args.workloads]
        for name, Ms in todo:
            if name != wl.name:
                gw.release()
                gw = GpuWorkload(q, WORKLOADS[name], dev)
            for Mi in Ms:
                r = gw.measure(Mi, args.steps, 3, world, min_s=MIN_TIMED_S)
                entries.append(entry_line(gw.wl, r, pk))
                del r
        gw.release()
        N_out, K = LINEAR_SHAPE
        for qt, gs, act in LINEAR_REPORTED:
            if args.workloads is not None and "linear" not in args.workloads:
                break
            gl = GpuLinear(q, qt, gs, act, N_out, K, dev)
            for Mi in LINEAR_MS:
                entries.append(gl.entry(Mi, gl.measure(Mi, args.steps, 3, min_s=MIN_TIMED_S), pk))
            gl.release()
    return wl, M, main, ms, e2e_ms, entries, pk


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        return run_reference(args)
    if args.record_traffic:
        return record_traffic(*args.record_traffic)
    if args.ncu_pass:
        return run_ncu_pass(args)
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    wl, M, main_r, ms, e2e_ms, entries, pk = run_gpu(args, rank, world)
    if rank == 0:
        import oracle  # noqa: F401  (CPU baseline leg only)
        layer_cpu = make_layer(wl, seed=0)
        n_tok, secs = oracle_sample(wl, layer_cpu, main_r["inp"], args.cpu_sample_s)
        del layer_cpu
        cpu_tps = n_tok / secs
        by = main_r["bytes"]
        roof, layer = roofline_entry(wl, M, ms, main_r["kernel_ms"], by, pk)
        roof["traffic"] = recorded_traffic(wl.name, M, roof["kernel"])
        roof["layer_frac_hbm"] = layer["frac_hbm_layer"]
        line = {
            "metric": METRIC,
            "value": whole_job_tokens_per_s(M, world, ms),
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": f"f16 MMA operands, f32 accumulate, {wl.qt} weights, {wl.act} activations",
            "data": "synthetic (seeded N(0,0.02) weights quantized offline, N(0,1) activations, random router)",
            "config": workload_config(wl, M),
            "tflops": world * layer["tflops"],
            "weight_gbs": world * layer["weight_gbs"],
            "roofline": roof,
            "layer": layer,
            "cpu_baseline": {"value": cpu_tps, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"float64 numpy oracle on the first {n_tok} of the {M} tokens "
                                       f"(each token dequantizes its {wl.k} experts), {secs:.1f} s"},
            "e2e": {"value": whole_job_tokens_per_s(M, world, e2e_ms), "unit": "tokens/s",
                    "h2d_bytes_per_step": int(M * wl.H * 2 + 2 * M * wl.k * 4),
                    "d2h_bytes_per_step": int(M * wl.H * 2), "ms_per_step": e2e_ms},
            "gpu_launches": int(round(main_r["launches_per_step"] * args.steps)),
            "clocks": main_r["clocks"],
            "kernel_ms": {n: round(v, 5) for n, v in main_r["kernel_ms"].items()},
            "workloads": entries,
        }
        line["config"]["l2"] = (f"inputs larger than L2: {by['weights'] / 1e6:.0f} MB of touched expert weights per "
                                f"step, rotated across {main_r['copies']} packed copies between steps (L2 129 MB); "
                                "each reported workload likewise")
        print(json.dumps(line))
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def run_ncu_pass(args):
    """Each reported (workload, M) runs 3 forwards on one packed copy (7 launches
    each, 2 of them GEMMs), in REPORTED order, and prints one JSON line per entry
    after its forwards, so a capture of the GEMM launches maps to entries by order."""
    import torch
    import weight_only_quantized_moe_gb300 as q
    q.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    for name, Ms in REPORTED:
        if args.workloads and name not in args.workloads:
            continue
        gw = GpuWorkload(q, WORKLOADS[name], dev)
        for M in Ms:
            if args.M and M != args.M:
                continue
            inp, x, ids, w = gw.inputs(M)
            out = torch.empty_like(x)
            ws = q.alloc_workspace(q.qmoe_workspace_size(gw.base, M, gw.wl.k), dev)
            for _ in range(3):
                q.qmoe_forward(gw.base, x, ids, w, out=out, workspace=ws)
            torch.cuda.synchronize()
            st = q.qmoe_read_device_status(ws)
            print(json.dumps({"ncu_pass": name, "M": M, "status": q.status_string(st),
                              "plan": q.qmoe_describe_plan(gw.base, M, gw.wl.k)}), flush=True)
            if st != q.QMOE_OK:
                raise RuntimeError(f"{name} M={M}: device status {q.status_string(st)}")
            del x, ids, w, out, ws
        gw.release()


def record_traffic(csv_path, pass_log):
    """profiles/dram_traffic.txt from a one-pass ncu capture of `--ncu-pass`: the
    GEMM launches come in entry order, 6 per entry (3 forwards x gate/up, down);
    the third forward's pair is recorded, with the current kernel-source hash."""
    import csv
    with open(csv_path) as f:
        rows = list(csv.reader([line for line in f if line.startswith('"')]))
    col = {h: i for i, h in enumerate(rows[0])}
    launch = {}
    for r in rows[1:]:
        launch.setdefault(int(r[col["ID"]]), {})[r[col["Metric Name"]]] = float(r[col["Metric Value"]])
    with open(pass_log) as f:
        entries = [json.loads(line) for line in f if line.startswith('{"ncu_pass"')]
    ids = sorted(launch)
    if len(ids) != 6 * len(entries):
        raise SystemExit(f"{len(ids)} GEMM launches for {len(entries)} entries (want 6 each)")
    h = kernel_source_hash()
    out = ["# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu capture,",
           "# read by bench.py for the roofline \"traffic\" field.  The fifth column is the first 16 hex",
           "# digits of sha256(gemm.cuh + ptx.cuh) of the kernel source that was captured; bench.py",
           "# reports null when the current source differs.  Commands (one pass per launch, cold L2):",
           "#   python bench.py --ncu-pass > pass.log 2>&1 && ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,"
           "gpu__time_duration.sum \\",
           "#       --clock-control none -k regex:qmoe_gemm --csv --print-units base --log-file traffic.csv "
           "python bench.py --ncu-pass > pass.log",
           "#   python bench.py --record-traffic traffic.csv pass.log",
           "# (each entry runs 3 forwards; the 3rd forward's gate/up and down launches are recorded)",
           "# workload M kernel bytes_per_launch source_sha256_16 read_bytes write_bytes duration_ns"]
    for n, e in enumerate(entries):
        for kname, lid in (("gemm_gate_up", ids[6 * n + 4]), ("gemm_down", ids[6 * n + 5])):
            g = launch[lid]
            rd, wr = int(g["dram__bytes_read.sum"]), int(g["dram__bytes_write.sum"])
            out.append(f'{e["ncu_pass"]} {e["M"]} {kname} {rd + wr} {h} {rd} {wr} {int(g["gpu__time_duration.sum"])}')
    with open(os.path.join(ROOT, "profiles", "dram_traffic.txt"), "w") as f:
        f.write("\n".join(out) + "\n")
    print(f"{len(out) - 9} launches recorded for source {h}")


def run_reference(args):
    wl = WORKLOADS[args.workload]
    M = args.M or (DEFAULT_M if DEFAULT_M in wl.Ms else wl.Ms[0])
    layer = make_layer(wl, seed=0)
    inp = make_inputs(wl, M, seed=0)
    budget = max(1.0, min(args.cpu_sample_s, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(wl, layer, inp, budget / 4)
    toks, secs = 0, 0.0
    for _ in range(args.steps):
        n, s = oracle_sample(wl, layer, inp, budget)
        toks += n
        secs += s
    v = toks / secs
    line = {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, M), "impl": "reference",
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"each step: float64 oracle on leading tokens of the M={M} batch for about "
                                       f"{budget:.1f} s; {toks} tokens in {secs:.1f} s"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
