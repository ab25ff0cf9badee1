"""bench.py's reference arm on the CPU: the fp64 oracle timed on the host cores, printing one JSON
line with the same metric, unit and config as the GPU arm, plus "impl": "reference", a
cpu_baseline describing the run and an e2e object with no host-device bytes."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_reference(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          *args], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", [None, "single_head_fp32"])
def test_reference_arm_line(workload):
    args = ["--steps", "2", "--warmup", "3"] + (["--workload", workload] if workload else [])
    d = run_reference(*args)
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "TFLOPS" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == (workload or "mha_N2048_d64")
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == d["value"]
    assert cpu["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
