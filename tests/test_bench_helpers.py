"""Host-side arithmetic of bench.py (no GPU): peaks, the derived FFMA peak,
the per-clock comparison of power-capped parts, and the shared config."""
import bench


def test_ffma_peak_from_clock():
    peaks = {"sm_max_mhz": 2070.0}
    # 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz
    assert abs(bench.fp32_ffma_peak(152, peaks) - 80.54784) < 1e-9


def test_per_clock_ratio():
    peaks = {"bf16_tflops_sustained": 1723.9, "sustained_sm_mhz": 1477.0}
    r = bench.per_clock(1614.7, {"sm_mhz": 1402.0}, peaks)
    assert abs(r["tflops_per_ghz"] - 1614.7 / 1.402) < 1e-9
    assert abs(r["sustained_tflops_per_ghz"] - 1723.9 / 1.477) < 1e-9
    assert abs(r["ratio"] - (1614.7 / 1.402) / (1723.9 / 1.477)) < 1e-12
    assert bench.per_clock(1614.7, {"sm_mhz": None}, peaks) is None
    assert bench.per_clock(1614.7, None, peaks) is None
    assert bench.per_clock(1614.7, {"sm_mhz": 1400.0}, {"bf16_tflops_sustained": 1.0}) is None


def test_both_arms_print_the_same_config():
    import inspect
    # both arms build their `config` from the same function
    assert "headline_config(" in inspect.getsource(bench.run_reference)
    assert "headline_config(" in inspect.getsource(bench.run_ours)
    assert bench.headline_config(1)["parallelism"] == "single GPU"
    assert bench.headline_config(8)["parallelism"] == "replicas"
    assert "4092" in bench.headline_config(1)["workload"]


def test_whole_job_throughput():
    # 2 ranks x 1 GFLOP per step x 10 steps over 20 ms = 1000 GFLOP/s
    assert abs(bench.whole_job_gflops(2, 1e9, 10, 20.0) - 1000.0) < 1e-9
