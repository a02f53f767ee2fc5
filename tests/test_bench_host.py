"""Host-side arithmetic of bench.py: the work counts its roofline divides by,
the rule that picks the tensor peak, and the gate that keeps a profiled
DRAM figure only while the kernel's sources are the ones it was taken on."""

import types

import bench
from ffn_block_gb300 import inputs as I


def _shape(name):
    return types.SimpleNamespace(**I.CONFIGS[name])


def test_step_flops_are_the_six_contractions():
    # 18 B T D H: GEMM1 forward, data and weight gradients (4 B T D H each)
    # and the same three for GEMM2 (2 B T D H each).
    for name in ("c1", "c2", "c3", "c4"):
        s = _shape(name)
        per_launch = bench.gemm_flops_per_launch(s)
        assert sum(per_launch.values()) == bench.flops_per_step(s)
        assert per_launch["gemm1_fwd"] == 2 * per_launch["gemm2_fwd"]


def test_minimum_bytes_at_the_production_shape():
    s = _shape("c3")
    # x, dy in; y, dx out (bf16), plus the parameters read twice and their
    # gradients written once.
    act = 4 * 1024 * 64 * 1280 * 2
    params = (3 * 64 * 1280 * 2560 + 64 * 2 * 2560 + 64 * 1280 + 6 * 1280 + 4 * 2560) * 2
    assert bench.min_bytes_per_step(s) == act + 3 * params
    assert abs(bench.min_bytes_per_step(s) - 4.45e9) < 0.01e9


def test_gate_backward_bytes_are_its_three_tensors():
    s = _shape("c3")
    n = 1024 * 64
    # dh (H) and Z (2H) read, dZ (2H) written, 16-bit.
    assert bench.row_bytes_per_launch(s)["gate_bwd"] == n * 5 * 2560 * 2


def test_peak_rule_burst_only_at_full_clock():
    peaks = {"bf16_tflops": 1932.8, "bf16_tflops_sustained": 1703.7}
    assert bench.tensor_peak(peaks, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0})[2] == "burst"
    assert bench.tensor_peak(peaks, {"sm_mhz": 1967.0, "sm_max_mhz": 2070.0})[2] == "burst"
    assert bench.tensor_peak(peaks, {"sm_mhz": 1957.0, "sm_max_mhz": 2070.0})[2] == "sustained"
    assert bench.tensor_peak(peaks, {"sm_mhz": None, "sm_max_mhz": None})[2] == "burst"
    burst, sustained, _ = bench.tensor_peak(peaks, {})
    assert (burst, sustained) == (1932.8, 1703.7)


def test_profiled_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "kern_work.md").write_text(
        "# a summary\n\n- source_hash: `abc123`\n- dram_bytes_per_launch: 123456\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # Taken on the current sources: the figure is used ...
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel=None: "abc123")
    assert bench.profiled_traffic("kern", "work") == 123456.0
    # ... none once the sources have changed, or without a summary.
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel=None: "def456")
    assert bench.profiled_traffic("kern", "work") is None
    assert bench.profiled_traffic("other", "work") is None


def test_source_hash_covers_the_kernel_and_shared_headers():
    # A GEMM launch name maps to the GEMM's sources; unknown names to all.
    assert bench.kernel_source_hash("gemm1_wgrad") == bench.kernel_source_hash("gemm2_fwd")
    assert bench.kernel_source_hash("gemm1_wgrad") != bench.kernel_source_hash("gate_bwd")
    assert len(bench.kernel_source_hash()) == 16
