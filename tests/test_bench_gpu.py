"""bench.py's GPU leg prints one JSON line with every key of its contract (a short run on the tiny workload)."""

import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")
def test_bench_json_contract():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny", "--steps", "3",
                        "--warmup", "3", "--cpu-budget", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks", "cpu_baseline"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] >= 3 and d["value"] > 0 and d["ms_per_step"] > 0
    assert d["unit"] == "GFLOP/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["vs_baseline"] is None and d["dtype"] == "f32" and d["data"] == "synthetic"
    assert d["config"]["workload"] == "tiny" and "l2" in d["config"]
    roof = d["roofline"]
    assert roof["bound"] in ("alu", "hbm") and roof["unit"] in ("TFLOP/s", "GB/s")
    assert roof["achieved"] > 0 and roof["peak"] > 0 and abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    assert "traffic" in roof
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "GFLOP/s"
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] >= 3 * 4   # T = 4 step launches per bench step, each timed bench step
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] > 0 and cpu["cores"] >= 1 and cpu["sample"]
    ctx = d["one_launch_context"]
    assert ctx["us_per_step"] > 0 and "context only" in ctx["note"]


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")
def test_chain_workloads_beside_the_headline():
    """The producer-chain and PDL-chain figures the large workload's line carries (measure_chain_workload), on a short
    run: per-step time, the fraction of the shape's roofline, the kernel, the clocks; the producer chain also carries
    the chain with the producer and the producer alone."""
    import argparse
    import sys as _sys
    _sys.path.insert(0, ROOT)
    import bench
    import fp32_gemm_gb300 as gx
    args = argparse.Namespace(steps=2, warmup=3, no_workspace=False)
    dev = torch.device("cuda", 0)
    for name in ("pdl_chain", "producer_chain"):
        d = bench.measure_chain_workload(gx, name, args, 1, 0, dev, torch.cuda.current_stream(), 0)
        assert d["us_per_step"] > 0 and 0 < d["frac_of_shape_roofline"] < 1.5 and d["gflops"] > 0
        assert d["kernel"].startswith("gx_") and d["roofline_bound"] in ("alu", "hbm")
        if name == "producer_chain":
            assert d["us_per_step_with_producer"] > 0 and d["producer_us_per_step"] > 0


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")
def test_trace_mode_prints_the_gap():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "pdl_chain", "--trace",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    t = json.loads(lines[0])["trace"]
    assert 0 < t["gap_us"]["mean"] < 50 and t["step_period_us"] > 0 and t["end_spread_us"] >= 0
    assert t["us_per_step_plain"] > 0 and t["us_per_step_traced"] > 0
