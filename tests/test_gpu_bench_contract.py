"""bench.py's output contract on one GPU: one JSON line with the keys the
benchmark harness reads, the timed value consistent with the per-step time,
and the roofline, CPU-baseline, end-to-end and clock records filled in."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    res = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=900)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, res.stdout[-2000:]
    return json.loads(lines[0])


def test_default_step_json_line():
    d = run_bench("--steps", "3", "--warmup", "3")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["unit"] == "TFLOP/s"
    # value = the step's work over the timed step time
    flops = 2 * 4096 ** 3 * 2
    assert d["value"] == pytest.approx(flops / (d["ms_per_step"] / 1e3) / 1e12, rel=1e-6)
    assert "workload" in d["config"]
    rl = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in rl, key
    assert 0.0 < rl["frac"] < 1.5 and rl["frac"] == pytest.approx(rl["achieved"] / rl["peak"])
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 4 * 4096 * 4096 * 2 + 2 * 4096 * 4096 * 2
    assert e2e["d2h_bytes_per_step"] == 4 * 4096 * 4096 + 2 * 4096 * 4096
    assert e2e["value"] < d["value"]  # the copies are inside the end-to-end region
    assert d["clocks"]["sm_max_mhz"] > 0 and isinstance(d["clocks"]["reasons"], list)
    assert d["gpu_launches"] == 2 * 3  # one SGEMM and one BF16 launch per timed step
    assert cb["cpu_model"] and cb["per_workload"]["sgemm_256"]["one_core_s"] > 0
    # the timed outputs and the other workloads against the oracle
    par = d["parity"]
    assert par["ok"] is True
    for name in ("sgemm_256", "sgemm_4096", "bf16_4096", "bf16_mlp_8192x14336x4096",
                 "bf16_decode_64x8192x8192"):
        rec = par["workloads"][name]
        assert rec["random"]["violations"] == 0 and rec["random"]["compared"] > 0, name
        assert rec["integer"]["mismatches"] == 0, name
    # the headline products are compared whole (the oracle finishes 4096^3 in seconds)
    assert par["workloads"]["bf16_4096"]["random"]["compared"] == 4096 * 4096
    for name, bound in (("sgemm_256", "alu"), ("bf16_mlp_8192x14336x4096", "tensor"),
                        ("bf16_decode_64x8192x8192", "hbm")):
        rl = d["rooflines"][name]
        assert rl["bound"] == bound and 0.0 < rl["frac"] < 1.5, name
        assert d["kernels"][name]["calls"] > 0
