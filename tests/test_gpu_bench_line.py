"""The bench's JSON line on a GPU: one small run of bench.py (one Llama-3.1-8B layer) must print one
line with every key of its contract, internally consistent: throughput against the step time, the
roofline fraction against its own numbers, the end-to-end figure with its copied bytes, the clocks,
the kernel count and a clean device status."""

import json
import subprocess
import sys

import pytest

import bench

pytestmark = pytest.mark.gpu


def test_bench_line_keys_and_consistency():
    r = subprocess.run([sys.executable, "bench.py", "--workload", "llama-3.1-8b", "--layers", "1", "--steps", "3",
                        "--warmup", "3", "--no-per-workload"], capture_output=True, text=True, timeout=900,
                       cwd=bench.ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks",
              "device_status", "step_ms", "graph_replay", "kernels"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["unit"] == "TFLOP/s" and line["dtype"] == "bf16"
    assert line["device_status"] == 0
    flops = line["config"]["ns_flops_per_step"]
    assert abs(line["value"] - flops / (line["ms_per_step"] * 1e-3) / 1e12) <= 1e-6 * line["value"]
    roof = line["roofline"]
    assert roof["bound"] in ("tensor", "hbm", "alu") and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert abs(roof["achieved"] - roof["work_per_launch"] / (roof["ms_per_launch"] * 1e-3) / 1e12) <= 1e-6 * roof["achieved"]
    assert 0.2 < roof["frac"] < 1.4, roof  # a one-layer set runs at the full clock, above the sustained peak
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] > 0 and cpu["cores"] >= 1 and cpu["sample"]
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "TFLOP/s" and e2e["returned_weights_match_device"] is True
    params = line["config"]["params"]
    assert e2e["h2d_bytes_per_step"] == 2 * params  # bf16 gradients
    assert e2e["d2h_bytes_per_step"] == 2 * params + 4  # bf16 weights and the status word
    assert line["gpu_launches"] == 3 * (2 + 3 * line["config"]["ns_steps"])
    assert line["clocks"]["sm_mhz"] > 0 and isinstance(line["clocks"]["reasons"], list)
    st = line["step_ms"]
    assert st["min"] <= st["median"] <= st["p90"] <= st["max"]
    assert line["graph_replay"]["device_status"] == 0 and line["graph_replay"]["ms_per_step"] > 0
