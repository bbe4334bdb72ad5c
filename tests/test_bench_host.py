"""Host-side pieces of bench.py that need no GPU: the kernel fingerprint that
ties the committed DRAM-traffic figures to the kernel code they were taken
on (so that they read null once the code changes), the per-step statistics,
and the bench's JSON contract for the reference arm."""

import json
import subprocess
import sys

import bench


def test_fingerprint_ignores_comments_but_not_code():
    a = "int f(int x) {\n  return x + 1;  // add one\n}\n"
    b = "/* header */\nint f(int x) {\n  // comment moved\n  return x + 1;\n}\n"
    c = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_traffic_is_null_for_unknown_workloads():
    assert bench.traffic_for("gemm", "no-such-workload") is None


def test_step_stats():
    st = bench.step_stats([5.0, 1.0, 4.0, 2.0, 3.0, 10.0, 6.0, 7.0, 8.0, 9.0, 11.0])
    assert st == {"median": 6.0, "p90": 10.0, "min": 1.0, "max": 11.0}
    assert bench.step_stats([]) is None
    assert bench.step_stats([2.5]) == {"median": 2.5, "p90": 2.5, "min": 2.5, "max": 2.5}


def test_reference_arm_line():
    # the oracle arm: one JSON line with the contract's keys, on the host cores
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "toy", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=bench.ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
