#!/usr/bin/env python
"""Benchmark of the fused weight-only-quantized MoE layer on GB300.

One step = one full layer forward (moe_align, token gather, gate/up GEMM with
fused SiLU*up, down GEMM with the routing weight, top-k reduce) over one batch
of M tokens of a synthetic workload shaped like the pages' models.  Prints ONE
JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--M M] [--no-sweep]

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
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--cpu-sample-s", type=float, default=20.0)
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


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
    """Samples the SM clock and the clock-event reasons of one GPU every ~2 ms
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
            time.sleep(0.002)

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
# GPU arm
# ----------------------------------------------------------------------------
def algorithmic_bytes(wl, dl, inp):
    """Bytes the method must move per layer call: the touched experts' packed
    weights and scales, x in, intermediate write + read, out."""
    d = len(np.unique(inp.topk_ids))
    M = inp.x.shape[0]
    P = M * wl.k
    per_expert_w13 = dl.w13.numel() // wl.E + (2 * wl.I * 4 if wl.qt == "int8" else 0)
    per_expert_w2 = dl.w2.numel() // wl.E + (wl.H * 4 if wl.qt == "int8" else 0)
    act = 2
    gemm1 = d * per_expert_w13 + P * wl.H * act + P * wl.I * act
    gemm2 = d * per_expert_w2 + P * wl.I * act + P * wl.H * 4
    total = d * (per_expert_w13 + per_expert_w2) + M * wl.H * act * 2 + 2 * P * wl.I * act
    return {"distinct_experts": d, "gemm_gate_up": gemm1, "gemm_down": gemm2, "layer": total,
            "weights": d * (per_expert_w13 + per_expert_w2)}


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


def run_gpu(args, rank, world):
    import torch

    import weight_only_quantized_moe_gb300 as q
    from weight_only_quantized_moe_gb300 import build as qbuild

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    qbuild.build()
    q.lib()
    wl = WORKLOADS[args.workload]
    M = args.M or (DEFAULT_M if DEFAULT_M in wl.Ms else wl.Ms[0])
    layer = make_layer(wl, seed=0)
    base = q.DeviceLayer.from_canonical(wl.qt, wl.act, layer.q13, layer.s13, layer.q2, layer.s2, layer.g13,
                                        layer.g2, device=dev)
    # rotate through copies of the packed weights so that no step finds them in L2
    copies = [base]
    n_copies = max(1, min(4, math.ceil(3 * L2_BYTES / max(1, base.weight_bytes())) + 1))
    for _ in range(n_copies - 1):
        copies.append(q.DeviceLayer(base.qt, base.E, base.H, base.I, base.act, base.w13.clone(), base.w2.clone(),
                                    None if base.s13 is None else base.s13.clone(),
                                    None if base.s2 is None else base.s2.clone(),
                                    None if base.perm13 is None else base.perm13.clone()))
    del layer
    stream = torch.cuda.current_stream()

    def measure(M, steps, warmup, profile=True):
        inp = make_inputs(wl, M, seed=0)
        x = torch.from_numpy(inp.x).to(base.torch_dtype).to(dev)
        ids = torch.from_numpy(inp.topk_ids).to(dev)
        w = torch.from_numpy(inp.topk_weights).to(dev)
        out = torch.empty_like(x)
        ws = q.alloc_workspace(q.qmoe_workspace_size(base, M, wl.k), dev)
        for i in range(warmup):
            q.qmoe_forward(copies[i % len(copies)], x, ids, w, out=out, workspace=ws)
        st = q.qmoe_read_device_status(ws)
        if st != q.QMOE_OK:
            raise RuntimeError(f"device status after warm-up: {q.status_string(st)}")
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(dev.index) as clk:
            e0.record(stream)
            for i in range(steps):
                q.qmoe_forward(copies[i % len(copies)], x, ids, w, out=out, workspace=ws)
            e1.record(stream)
            torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        res = {"M": M, "ms": ms, "clocks": clk.summary(), "inp": inp}
        if profile:
            # second pass over the same K steps with CUDA events around each kernel launch
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(LAUNCH_NAMES))] for _ in range(steps)]
            launches = 0
            for i in range(steps):
                launches += q.qmoe_forward_profiled(copies[i % len(copies)], x, ids, w, out, ws, evs[i])
            torch.cuda.synchronize()
            per = {}
            for j, name in enumerate(LAUNCH_NAMES):
                per[name] = sum(evs[i][2 * j].elapsed_time(evs[i][2 * j + 1]) for i in range(steps)) / steps
            res["kernel_ms"] = per
            res["launches_per_step"] = launches / steps
        st = q.qmoe_read_device_status(ws)
        if st != q.QMOE_OK:
            raise RuntimeError(f"device status: {q.status_string(st)}")
        res["bytes"] = algorithmic_bytes(wl, base, inp)
        res["copies"] = len(copies)
        res["x"], res["ids"], res["w"] = x, ids, w
        return res

    main = measure(M, args.steps, args.warmup)
    ms = max_over_ranks(main["ms"], world, dev)

    # end to end through the host-buffer entry point: pinned H2D of x/ids/weights,
    # the forward, D2H of out, every step
    xh = main["x"].cpu().pin_memory()
    idh = main["ids"].cpu().pin_memory()
    wh = main["w"].cpu().pin_memory()
    outh = torch.empty_like(xh).pin_memory()
    wsh = q.alloc_workspace(q.qmoe_workspace_size_host(base, M, wl.k), dev)
    for i in range(args.warmup):
        q.qmoe_forward_host(copies[i % len(copies)], xh, idh, wh, outh, wsh)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        q.qmoe_forward_host(copies[i % len(copies)], xh, idh, wh, outh, wsh)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)

    sweep = []
    if not args.no_sweep and rank == 0:
        for Ms in wl.Ms:
            if Ms == M:
                continue
            r = measure(Ms, max(5, args.steps // 5), 3)
            sweep.append(r)
    return wl, M, main, ms, e2e_ms, sweep, base


def summarize(wl, r, hbm, tc):
    M = r["M"]
    ms = r["ms"]
    k = r["kernel_ms"]
    by = r["bytes"]
    flops = wl.flops(M)
    return {"M": M, "ms": round(ms, 5), "tokens_per_s": M / (ms * 1e-3),
            "tflops": flops / (ms * 1e-3) / 1e12,
            "weight_gbs": by["weights"] / (ms * 1e-3) / 1e9,
            "hbm_frac_layer": by["layer"] / (ms * 1e-3) / 1e9 / hbm,
            "distinct_experts": by["distinct_experts"],
            "kernel_ms": {n: round(v, 5) for n, v in k.items()}}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        return run_reference(args)
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    wl, M, main_r, ms, e2e_ms, sweep, base = run_gpu(args, rank, world)
    hbm, tc_burst, tc_sust, peak_src = peaks()
    if rank == 0:
        import oracle  # noqa: F401  (CPU baseline leg only)
        layer_cpu = make_layer(wl, seed=0)
        n_tok, secs = oracle_sample(wl, layer_cpu, main_r["inp"], args.cpu_sample_s)
        cpu_tps = n_tok / secs
        by = main_r["bytes"]
        kms = main_r["kernel_ms"]
        dominant = max(("gemm_gate_up", "gemm_down"), key=lambda n: kms[n])
        flops = wl.flops(M)
        # the dominant GEMM's roofline: HBM (weight stream) or tensor pipe, by its
        # arithmetic intensity against the measured peaks' ratio
        P = M * wl.k
        kflops = 2.0 * P * (2 * wl.I if dominant == "gemm_gate_up" else wl.I) * wl.H
        kms_s = kms[dominant] * 1e-3
        if kflops / by[dominant] > tc_burst * 1e12 / (hbm * 1e9):
            roof = {"bound": "tensor", "achieved": kflops / kms_s / 1e12, "peak": tc_burst, "unit": "TFLOP/s",
                    "frac": kflops / kms_s / 1e12 / tc_burst,
                    "peak_source": f"{peak_src} bf16_tflops burst (MEASURED_PEAKS.json cuBLAS bf16 GEMM; "
                                   "the f16 MMAs run at the bf16 rate)",
                    "algorithmic_flops_per_launch": kflops}
        else:
            roof = {"bound": "hbm", "achieved": by[dominant] / kms_s / 1e9, "peak": hbm, "unit": "GB/s",
                    "frac": by[dominant] / kms_s / 1e9 / hbm,
                    "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json copy bandwidth)",
                    "algorithmic_bytes_per_launch": by[dominant]}
        roof.update({"kernel": dominant, "traffic": recorded_traffic(wl.name, M, dominant),
                     "layer_frac_hbm": by["layer"] / (ms * 1e-3) / 1e9 / hbm})
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
            "dtype": f"{wl.act} MMA operands, f32 accumulate, {wl.qt} weights",
            "data": "synthetic (seeded N(0,0.02) weights quantized offline, N(0,1) activations, random router)",
            "config": workload_config(wl, M),
            "tflops": world * flops / (ms * 1e-3) / 1e12,
            "weight_gbs": world * by["weights"] / (ms * 1e-3) / 1e9,
            "roofline": roof,
            "cpu_baseline": {"value": cpu_tps, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"float64 numpy oracle on the first {n_tok} of the {M} tokens "
                                       f"(each token dequantizes its {wl.k} experts), {secs:.1f} s"},
            "e2e": {"value": whole_job_tokens_per_s(M, world, e2e_ms), "unit": "tokens/s",
                    "h2d_bytes_per_step": int(M * wl.H * 2 + 2 * M * wl.k * 4),
                    "d2h_bytes_per_step": int(M * wl.H * 2), "ms_per_step": e2e_ms},
            "gpu_launches": int(round(main_r["launches_per_step"] * args.steps)),
            "clocks": main_r["clocks"],
            "kernel_ms": {n: round(v, 5) for n, v in kms.items()},
            "sweep": [summarize(wl, r, hbm, tc_burst) for r in sweep],
        }
        line["config"]["l2"] = (f"inputs larger than L2: {by['weights'] / 1e6:.0f} MB of touched expert weights per "
                                f"step, rotated across {main_r['copies']} packed copies between steps (L2 129 MB)")
        print(json.dumps(line))
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


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
