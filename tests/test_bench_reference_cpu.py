"""bench.py's reference arm (the oracle on the host cores, no GPU): one JSON
line with the base contract's keys, the decode workload's config and a
positive throughput, within a small time budget."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_its_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3", "--warmup", "3",
                          "--ref-budget-s", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["config"]["workload"] == "llama7b_decode_g128_r32" and line["config"]["calls_per_step"] == 12
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_rotates_calls_when_a_step_cannot_hold_all_twelve():
    """With a per-step share of the time smaller than one row of each of the
    12 calls, each step times a rotating block of the calls; the line stays
    well formed and the run stays short."""
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "60", "--warmup", "3",
                          "--ref-budget-s", "0.05"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["steps"] == 60 and line["value"] > 0
    assert "in rotation" in line["cpu_baseline"]["sample"]
