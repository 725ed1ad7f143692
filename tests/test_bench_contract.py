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
