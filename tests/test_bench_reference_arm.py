"""bench.py's reference arm on the host cores: `--impl reference` times the fp64 oracle
on a bounded sample of the bench workload and prints one JSON line with the same metric,
unit and workload description as the GPU arm, plus its own cpu_baseline and e2e. Runs without a GPU;
this checks the line's contract, not the number."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["steps"] == 1 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["unit"] == "GB/s"
    sys.path.insert(0, ROOT)
    import bench
    # the GPU arm prints bench_config(workload, world): the same keys and values
    assert d["config"] == bench.bench_config(bench.DEFAULT_WORKLOAD, 1)
    assert d["config"]["workload"] == "add_rmsnorm_32768x4096"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
