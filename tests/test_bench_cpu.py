"""bench.py's CPU legs: the reference arm (the oracle timed on the host) prints one valid JSON line; the kernel-source
hash that guards the stored DRAM-traffic figure is stable."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "3", "--ref-seconds", "0.3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == (os.cpu_count() or 1)
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["warmup"] >= 3 and d["higher_is_better"] is True


def test_kernel_sha_is_stable():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.kernel_sha() == bench.kernel_sha() and len(bench.kernel_sha()) == 16
