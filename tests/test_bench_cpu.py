"""bench.py's byte accounting and its CPU reference arm (no GPU)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_algorithmic_bytes():
    m, _ = bench.workload("qkv_gate_set", 1)
    # 2 x 15,335,424 (Q4_K 4096x6656) + 2 x 256*26*210 + x once + 4 outputs
    assert bench.algorithmic_bytes(m, 1) == (
        2 * 15335424 + 2 * 256 * 26 * 210 + 4 * 6656 + 4 * 8704)
    assert bench.algorithmic_bytes(m, 1) == 33527808
    m, _ = bench.workload("q4k_4096", 8)
    assert bench.algorithmic_bytes(m, 8) == 15335424 + 8 * 4 * (6656 + 4096)
    m, _ = bench.workload("cat_q6k_q5k", 1)
    assert bench.algorithmic_bytes(m, 1) == 1075200 + 901120 + 2 * 4 * 2560 + 2 * 4 * 512


def test_reference_arm_json():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
         "reference", "--steps", "4", "--warmup", "3"],
        capture_output=True, text=True, check=True, timeout=300)
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["config"]["workload"] == "qkv_gate_set"
