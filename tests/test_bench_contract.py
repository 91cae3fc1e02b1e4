"""The bench's JSON contract on the host: the reference arm (the fp64 oracle
on the host cores) prints one line with the keys the driver reads, and the
helpers that turn per-launch times into the line's figures behave as stated.
No GPU is needed."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "1"], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOPS" and d["higher_is_better"] is True
    assert d["config"]["workload"] == bench.WORKLOAD
    assert d["steps"] == 1 and d["warmup"] >= 3  # the timing rules' minimum warm-up
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_geomean():
    assert bench.geomean([2.0, 8.0]) == pytest.approx(4.0)
    assert bench.geomean([5.0]) == pytest.approx(5.0)


def test_kernel_hash_ignores_comments():
    # The committed DRAM-traffic summary stays valid across comment-only
    # edits of the kernel sources, and not across code edits.
    code = "int f() { return 1; }  // one\n/* two */\n"
    assert bench._code_only(code) == bench._code_only("int f() { return 1; }\n")
    assert bench._code_only(code) != bench._code_only("int f() { return 2; }\n")
