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
