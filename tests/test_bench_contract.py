"""bench.py's JSON line, checked on the host (no GPU): the reference arm runs
the fp64 oracle on the CPU, so its line can be produced and checked here;
argument rules that hold for both arms are checked too."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_complete_json_line():
    r = _run("--impl", "reference", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline",
              "e2e"):
        assert k in d, k
    assert d["impl"] == "reference"
    assert d["unit"] == "TFLOP/s" and d["value"] > 0 and d["ms_per_step"] > 0
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"]["workload"] == "mlp_b2_s2048_h4096_hp16384_N2"
    # the main arm prints the same config object (bench.workload_config)
    import bench
    assert d["config"] == bench.workload_config("mlp_b2_s2048_h4096_hp16384_N2", 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_fewer_than_three_warmup_steps_are_refused():
    for impl in ("ours", "reference"):
        r = _run("--impl", impl, "--steps", "3", "--warmup", "2")
        assert r.returncode == 2 and "warmup" in r.stderr


def test_roofline_achieved_recomputes_from_the_per_call_time():
    """`achieved` is the work of one call divided by the kernel's device time
    per call (its launches in the call summed), and the line says how many
    launches a call holds, so a reader can recompute it from the line alone."""
    import bench

    class FakeBench:
        name = "no_such_workload"

        @staticmethod
        def kernel_work():
            return {"gemm_two": ("tensor", 2.0e12), "rows": ("hbm", 4.0e8)}

    # 10 calls of two launches in 12.5 ms; 10 calls of one launch in 0.5 ms
    prof = {"gemm_two": (10, 20, 12.5), "rows": (10, 10, 0.5)}
    peaks = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0, "hbm_gbs": 8000.0}
    top, kernels = bench.roofline_for(None, FakeBench, prof, peaks, "measured", sustained=False)
    assert top["kernel"] == "gemm_two" and top["kernel_launches_per_call"] == 2
    assert abs(top["avg_us"] - 1250.0) < 1e-9
    assert abs(top["achieved"] - 2.0e12 / (top["avg_us"] * 1e-6) / 1e12) < 1e-9
    assert abs(top["frac"] - top["achieved"] / 2000.0) < 1e-12
    assert top["traffic"] is None  # no committed counters for this workload
    assert "bf16_tflops" in top["peak_source"] and "sustained" not in top["peak_source"]
    rows = {k["kernel"]: k for k in kernels}
    assert abs(rows["rows"]["achieved"] - 4.0e8 / 50e-6 / 1e9) < 1e-9 and rows["rows"]["unit"] == "GB/s"
    assert abs(sum(k["share"] for k in kernels) - 1.0) < 1e-12
