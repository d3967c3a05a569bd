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


def test_clock_sampler_parses_smi_lines():
    # the sampler's parser on lines in nvidia-smi's csv,noheader,nounits format: median SM clock,
    # max clock, max power, and every throttle reason that was active in any sample
    sys.path.insert(0, ROOT)
    import bench
    s = bench.ClockSampler(0)
    s.source = "test"
    s._parse_smi("\n".join([
        "0, 1395, 2032, 612.40, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1410, 2032, 598.10, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1650, 2032, 420.00, 0x0000000000000000, Not Active, Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2032, 400.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]))
    out = s.summary()
    assert out["samples"] == 3 and out["sm_mhz"] == 1410.0 and out["sm_max_mhz"] == 2032.0
    assert out["power_w_max"] == 612.40
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
