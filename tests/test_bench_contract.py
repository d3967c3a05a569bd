"""The benchmark's reference arm (the fp64 oracle on the host cores) keeps the
JSON-line contract: one line from rank 0 with the metric, unit, value, the
CPU-baseline and end-to-end objects; other ranks print nothing and exit 0.
Runs bench.py as a subprocess on the small d2 workload (no GPU needed)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(extra_env=None, *args):
    env = dict(os.environ)
    env.update(extra_env or {})
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                         env=env, cwd=ROOT, timeout=600)
    return out


def test_reference_arm_prints_one_contract_line():
    out = run_bench(None, "--impl", "reference", "--steps", "2", "--warmup", "1", "--workload", "d2")
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["value"] > 0 and d["ms_per_step"] > 0
    assert d["metric"].startswith("Muon optimizer step")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_reference_arm_on_a_non_zero_rank_is_silent():
    out = run_bench({"RANK": "1", "WORLD_SIZE": "2"}, "--impl", "reference", "--steps", "1", "--warmup", "0",
                    "--workload", "d2")
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == ""
