"""The benchmark's one-line JSON contract on a GPU: a short run of bench.py (the
headline decode step plus the tiny fp32 workload) and every field the line must
carry, with values that make sense for one GB300."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def line():
    cmd = [sys.executable, "bench.py", "--steps", "3", "--warmup", "3", "--workloads", "c1", "--workload-reps", "3",
           "--ramp-steps", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    return json.loads(lines[0])


def test_headline_fields(line):
    assert line["metric"] and line["unit"] == "GB/s"
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["vs_baseline"] is None
    assert line["dtype"] == "bf16" and line["data"] == "synthetic"
    assert line["config"]["workload"] and "l2" in line["config"]
    assert line["device_status"] == 0


def test_roofline(line):
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert rf["achieved"] > 0 and rf["peak"] > 0
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"])
    assert 0.0 < rf["frac"] < 1.5  # a plain copy is the denominator: a little above 1 is possible, far above is not
    assert rf["traffic"] is None or rf["traffic"] > 0


def test_cpu_baseline_and_e2e(line):
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"] and cb["unit"]
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0


def test_launches_and_clocks(line):
    assert line["gpu_launches"] >= line["steps"]
    ck = line["clocks"]
    assert ck["sm_max_mhz"] > 0 and "reasons" in ck


def test_tiny_fp32_workload(line):
    w = line["workloads"]["tiny_decode_fp32"]
    assert w["ms"] > 0 and w["graph_ms"] > 0
