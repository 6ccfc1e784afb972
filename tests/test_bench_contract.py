"""The benchmark's output line, checked on CPU through its reference arm.

`bench.py --impl reference` times the fp64 oracle on the host cores and needs
no GPU, so the line it prints can be held to the benchmark's contract here:
exactly one JSON line on stdout, the metric of the measured arm, a positive
value, a `cpu_baseline` that describes the run and an `e2e` with no copies.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def _common(line, metric, unit, workload):
    assert line["impl"] == "reference"
    assert line["metric"] == metric and line["unit"] == unit
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["n_gpus"] == 1 and line["steps"] == 2 and line["warmup"] == 1
    assert line["ms_per_step"] > 0
    assert line["dtype"] == "f64" and line["data"] == "synthetic"
    assert line["config"]["workload"] == workload
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == line["value"] and cpu["unit"] == unit
    assert cpu["cores"] >= 1 and cpu["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == unit
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_attention_line():
    w = bench.workload_of("c1")
    line = _run("--impl", "reference", "--workload", "c1", "--steps", "2", "--warmup", "1")
    _common(line, bench.METRIC, "TFLOPS", w.name)
    assert line["config"]["Nq"] == w.Nq and line["config"]["d"] == w.d


@pytest.mark.parametrize("name", ["softmax_f32"])
def test_reference_arm_softmax_line(name):
    sw = bench.SOFTMAX_ALIASES[name]
    line = _run("--impl", "reference", "--workload", name, "--steps", "2", "--warmup", "1")
    assert line["unit"] == "GB/s"
    _common(line, line["metric"], "GB/s", sw.name)
    assert "softmax" in line["metric"]


def test_reference_arm_backward_line():
    w = bench.workload_of("c1")
    line = _run("--impl", "reference", "--workload", "c1:bwd", "--steps", "2", "--warmup", "1")
    _common(line, bench.BWD_METRIC, "TFLOPS", w.name + ":bwd")


def test_reference_arm_fp8_line():
    name = "custom:1,2,256,256,128"
    w = bench.workload_of(name)
    line = _run("--impl", "reference", "--workload", name + ":fp8", "--steps", "2", "--warmup", "1")
    _common(line, bench.FP8_METRIC, "TFLOPS", w.name + ":fp8")
    assert line["cpu_baseline"]["cores"] == 1
