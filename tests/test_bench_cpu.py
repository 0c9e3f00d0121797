"""The benchmark's reference arm (the CPU oracle on bounded samples) runs
without a GPU and prints one JSON line in the benchmark's contract."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["unit"] == "positions/s"
    assert line["config"]["workload"] == "full_decode_tile"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["steps"] == 1 and line["warmup"] == 3


def test_reference_arm_width_workload():
    """The verify-width workload's reference arm: the oracle's width verify,
    positions counted as the sum of (w + 1)."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--workload", "decode_verify_tile_width", "--cpu-seconds", "2"],
                         capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["config"]["workload"] == "decode_verify_tile_width"
    assert "verify_width" in line["config"] and line["config"]["verified_rows"] < 64 * 6
    assert line["value"] > 0 and "w + 1 rows" in line["cpu_baseline"]["sample"]


def _reference_line(workload):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--workload", workload, "--cpu-seconds", "2"],
                         capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    return json.loads(out.stdout.strip().splitlines()[-1])


def test_reference_arm_rnn_and_sts_workloads():
    line = _reference_line("rnn_decode_tile")
    assert line["config"]["sequential_head"].startswith("RNN") and line["value"] > 0
    line = _reference_line("sts_fit")
    assert line["config"]["workload"] == "sts_fit" and line["config"]["pairs"] == 4_194_304 * 7
    assert line["value"] > 0 and "bisection" in line["cpu_baseline"]["sample"]
