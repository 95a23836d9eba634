"""Host-side pieces of bench.py (no GPU): the recorded-traffic lookup and the
whole-job arithmetic."""
import os

import bench


def test_recorded_traffic_matches_current_source_only(tmp_path, monkeypatch):
    cur = bench.kernel_source_hash()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic.txt").write_text(
        "# comment\n"
        f"wl_a 16 gemm_gate_up 1234 {cur} x.md\n"
        f"wl_b 16 gemm_gate_up 999 0000000000000000 y.md\n")
    src = tmp_path / "weight_only_quantized_moe_gb300" / "csrc"
    src.mkdir(parents=True)
    for f in ("gemm.cuh", "ptx.cuh"):
        (src / f).write_bytes(open(os.path.join(bench.ROOT, "weight_only_quantized_moe_gb300", "csrc", f), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("wl_a", 16, "gemm_gate_up") == 1234
    assert bench.recorded_traffic("wl_a", 16, "gemm_down") is None
    assert bench.recorded_traffic("wl_a", 1, "gemm_gate_up") is None
    assert bench.recorded_traffic("wl_b", 16, "gemm_gate_up") is None  # captured from other source


def test_whole_job_tokens_per_s():
    assert bench.whole_job_tokens_per_s(16, 1, 1.0) == 16000.0
    assert bench.whole_job_tokens_per_s(16, 4, 2.0) == 32000.0


def test_algorithmic_bytes_and_roofline_arithmetic():
    from synth import WORKLOADS
    import numpy as np
    wl = WORKLOADS["mixtral8x7b_w4"]
    M = 4
    ids = np.array([[0, 1], [1, 2], [0, 2], [5, 1]], np.int32)
    w13, w2 = 1000, 500
    by = bench.algorithmic_bytes(wl, w13, w2, ids, M)
    assert by["distinct_experts"] == 4
    P = M * wl.k
    assert by["weights"] == 4 * (w13 + w2)
    assert by["gemm_gate_up"] == 4 * w13 + P * wl.H * 2 + P * wl.I * 2
    assert by["gemm_down"] == 4 * w2 + P * wl.I * 2 + P * wl.H * 4
    assert by["layer"] == 4 * (w13 + w2) + 2 * M * wl.H * 2 + 2 * P * wl.I * 2
    pk = {"hbm": 1000.0, "tc_burst": 2000.0, "tc_sust": 1800.0, "src": "test"}
    # weight-stream bound: 1e9 bytes in 2 ms -> 500 GB/s -> 0.5 of a 1000 GB/s peak
    by = {"gemm_gate_up": 1e9, "gemm_down": 1e8, "layer": 2e9, "weights": 1.5e9, "distinct_experts": 8}
    roof, layer = bench.roofline_entry(wl, 1, 4.0, {"gemm_gate_up": 2.0, "gemm_down": 1.0}, by, pk)
    assert roof["bound"] == "hbm" and roof["kernel"] == "gemm_gate_up"
    assert abs(roof["frac"] - 0.5) < 1e-12
    assert abs(layer["frac_hbm_layer"] - 0.5) < 1e-12 and abs(layer["frac_hbm_weights"] - 0.375) < 1e-12
    # a compute-heavy launch is judged against the tensor peak
    Mb = 8192
    by = {"gemm_gate_up": 1e9, "gemm_down": 5e8, "layer": 2e9, "weights": 1e9, "distinct_experts": 8}
    roof, layer = bench.roofline_entry(wl, Mb, 10.0, {"gemm_gate_up": 6.0, "gemm_down": 3.0}, by, pk)
    fl = bench.gemm_flops(wl, Mb, "gemm_gate_up")
    assert roof["bound"] == "tensor" and abs(roof["achieved"] - fl / 6e-3 / 1e12) < 1e-6
    assert abs(roof["frac_of_sustained_peak"] * 1800.0 - roof["achieved"]) < 1e-9
    assert layer["binding"] == "tensor"


def test_recorded_dram_traffic_matches_the_kernel_source():
    """Every line of profiles/dram_traffic.txt was captured from the current GEMM
    source (its hash column), and every (workload, M) the benchmark reports has
    both GEMM launches recorded, so the bench line's roofline.traffic is never
    null for a stale reason."""
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic.txt")
    h = bench.kernel_source_hash()
    seen = set()
    with open(path) as f:
        for line in f:
            p = line.split()
            if not p or p[0].startswith("#"):
                continue
            assert p[4] == h, f"{p[0]} M={p[1]} {p[2]}: captured from source {p[4]}, current {h}"
            assert int(p[3]) > 0
            seen.add((p[0], int(p[1]), p[2]))
    for name, Ms in bench.REPORTED:
        for M in Ms:
            for k in ("gemm_gate_up", "gemm_down"):
                assert (name, M, k) in seen, (name, M, k)
