"""bench.py's JSON line on a GPU: one line with every key of the benchmark
contract, consistent with itself (launch count, e2e byte counts, roofline
fraction), and the roofline's DRAM traffic taken from the committed ncu record
exactly when that record was made on the current kernel sources."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_has_the_contract_keys():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3", "--no-per-shape",
           "--no-cpu-baseline"]
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["higher_is_better"] is False
    assert d["value"] > 0 and d["unit"] == "ms" and d["dtype"] == "bf16"
    assert d["config"]["workload"] == "experts_128x1536x2048"
    assert d["gpu_launches"] == 3 * d["launches_per_step"] == 3 * 16
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == "ms" and e["equals_device_result"] is True
    assert e["h2d_bytes_per_step"] == e["d2h_bytes_per_step"] == 128 * 1536 * 2048 * 2
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["achieved"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        recorded = json.load(f)["source_hash"]
    if recorded == d["kernel_source_hash"]:
        assert r["traffic"] is not None and r["traffic"] > 0
    else:
        assert r["traffic"] is None and "changed" in r["traffic_note"]
    assert d["device_error_word"] == 0 and d["parity"]["rel_fro_err_vs_fp64_oracle"] <= d["parity"]["tolerance"]
