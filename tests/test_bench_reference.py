"""bench.py --impl reference (the CPU oracle timed as the reference arm) runs
on CPU and prints one JSON line of the contract."""
from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "nvfp4_128x128x256_f32", "--steps", "2", "--warmup", "3",
                        "--ref-step-s", "0.05"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["value"] > 0 and res["unit"] == "TFLOP/s"
    assert res["cpu_baseline"]["kind"] == "oracle" and res["cpu_baseline"]["cores"] >= 1
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["config"]["workload"] == "nvfp4_128x128x256_f32"
