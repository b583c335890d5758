"""bench.py's JSON line against the benchmark contract: the reference arm (the CPU oracle,
host cores only) here, and our arm on a B300 (`-m gpu`). Both run the tiny fp32 layer so
that a run takes seconds."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
COMMON = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
          "vs_baseline", "dtype", "data", "config")


def _run(*args, timeout=600):
    out = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True,
                         timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def _common(j, steps, warmup):
    for k in COMMON:
        assert k in j, k
    assert j["value"] > 0 and j["ms_per_step"] > 0
    assert (j["steps"], j["warmup"], j["n_gpus"]) == (steps, warmup, 1)
    assert j["higher_is_better"] is True and j["unit"] == "tokens/s"
    assert j["config"]["workload"] == "tiny_fp32"


def test_reference_arm_line():
    j = _run("--impl", "reference", "--config", "tiny_fp32", "--steps", "2", "--warmup", "1")
    _common(j, 2, 1)
    assert j["impl"] == "reference"
    # a step routes every token and computes the outputs of a token sample, which the
    # value counts
    assert "routing of all" in j["cpu_baseline"]["sample"]
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == j["value"]
    e2e = j["e2e"]
    assert e2e["value"] == j["value"] and e2e["unit"] == j["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_our_arm_line():
    j = _run("--config", "tiny_fp32", "--workloads", "none", "--no-variants", "--steps", "5", "--warmup", "3",
             "--cpu-seconds", "1")
    _common(j, 5, 3)
    assert "impl" not in j or j["impl"] != "reference"
    # value = the batch's tokens over the time per step
    assert j["value"] == pytest.approx(j["config"]["T"] / (j["ms_per_step"] / 1e3), rel=1e-6)
    r = j["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-6)
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    e2e = j["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == j["unit"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    # the forward's kernels every timed step, and those of the stage-event graphs run
    # between the timed steps when the run records stage times that way
    import bench
    import workloads as W
    per = bench.launches_per_forward(W.WORKLOADS["tiny_fp32"])
    assert j["gpu_launches"] in (per * 5, 2 * per * 5)
    c = j["clocks"]
    assert c["sm_max_mhz"] > 0 and isinstance(c["reasons"], list)
