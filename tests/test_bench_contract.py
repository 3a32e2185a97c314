"""The benchmark's reference arm on the CPU: one JSON line with the
contract's keys, timed on the float64 oracle, and the same `config` object
the GPU arm reports for the workload (no GPU needed)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
         "--workload", "c1_n512_d2", "--steps", "2", "--warmup", "1"],
        capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["h2d_bytes_per_step"] == 0
    sys.path.insert(0, ROOT)
    import bench
    from streaming_sinkhorn_solver_gb300.workloads import WORKLOADS
    assert line["config"] == json.loads(json.dumps(bench.arm_config(WORKLOADS["c1_n512_d2"])))
    assert line["metric"] == bench.METRIC


@pytest.mark.parametrize("name", ["c1_n512_d2", "c4_n50k_d512", "bs_n1m_d3"])
def test_arm_config_names_the_workload(name):
    import bench
    from streaming_sinkhorn_solver_gb300.workloads import WORKLOADS
    w = WORKLOADS[name]
    cfg = bench.arm_config(w)
    assert cfg["workload"] == name and (cfg["n"], cfg["m"], cfg["d"]) == (w.n, w.m, w.d)
    assert "model" not in cfg
    assert ("tau" in cfg) == (w.tau > 0)


def test_tensor_peak_scales_with_the_run_clock():
    """The tensor roofline's denominator is the measured sustained rate scaled
    from the clock it was measured at to the run's clock: a kernel that ran
    at 1800 MHz doing 1750 TFLOP/s against a 1745.7 TFLOP/s measurement at
    1500 MHz is at 0.83 of it, not above 1 (a fraction above 1 would be an
    accounting error, not a result)."""
    import bench
    peaks = {"bf16_tflops": 1925.9, "bf16_tflops_sustained": 1745.7, "source": "measured",
             "clocks_under_load": {"sm_mhz_median": 1500.0}}
    peak, src = bench.tensor_peak(peaks, 1800.0)
    assert abs(peak - 1745.7 * 1.2) < 1e-9 and "1800" in src
    assert 1750.0 / peak < 1.0
    same, _ = bench.tensor_peak(peaks, 1500.0)
    assert same == 1745.7
    burst, src = bench.tensor_peak({"bf16_tflops": 1925.9, "bf16_tflops_sustained": 1700.0,
                                    "source": "fallback"}, 1800.0)
    assert burst == 1925.9 and "burst" in src


def test_metric_points_cover_every_configuration_with_long_regions():
    import bench
    from streaming_sinkhorn_solver_gb300.workloads import WORKLOADS
    dense = {n for n, w in WORKLOADS.items() if w.tau == 0}
    assert dense == set(bench.METRIC_POINTS) | {bench.DEFAULT_WORKLOAD}
    assert bench.point_steps(300.0) == bench.POINT_MIN_STEPS
    assert bench.point_steps(1.0) * 1.0 >= bench.POINT_MIN_MS
    assert bench.point_steps(1e-6) == bench.POINT_MAX_STEPS


def test_kernel_source_hash_ignores_comments_only():
    """The committed ncu summaries stay attached to their kernels through
    comment edits, and detach on any code change."""
    import bench
    code = "int f(int x) {\n  return x + 1;  // one more\n}\n/* block\n comment */\n"
    assert bench._code_only(code) == bench._code_only(
        "int f(int x) {\n\n    return x + 1;   // another comment\n}\n")
    assert bench._code_only(code) != bench._code_only("int f(int x) {\n  return x + 2;\n}\n")

