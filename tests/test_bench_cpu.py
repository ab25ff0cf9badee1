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


@pytest.mark.parametrize("workload", [None, "single_head_fp32", "bwd_causal_N4096_d128"])
def test_reference_arm_line(workload):
    args = ["--steps", "2", "--warmup", "3"] + (["--workload", workload] if workload else [])
    d = run_reference(*args)
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "TFLOPS" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == (workload or "causal_N8192_d128")
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == d["value"]
    assert cpu["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_default_line_per_config_covers_the_other_specified_workloads():
    import bench
    from exact_attention_fa_gb300 import workloads as wl
    assert bench.DEFAULT_WORKLOAD == "causal_N8192_d128"
    assert bench.bench_workload(bench.DEFAULT_WORKLOAD).backward is False
    names = bench.per_config_names(bench.DEFAULT_WORKLOAD)
    assert names == ["single_head_fp32", "mha_N2048_d64", "blocksparse_N16384_d64",
                     "bwd_causal_N4096_d128"]
    assert set(names) | {bench.DEFAULT_WORKLOAD} == set(wl.SPECIFIED)


def test_oracle_sample_work_matches_the_metric():
    """The oracle's row-sampled tasks account exactly the metric's work: a full sweep of every
    (head, row offset) pair sums to the workload's algorithmic FLOPs."""
    import bench
    from exact_attention_fa_gb300 import workloads as wl
    for w in (wl.Workload("s_dense", 1, 2, 1024, 64, seed=1),
              wl.Workload("s_causal", 1, 2, 1024, 64, causal=True, seed=2),
              wl.Workload("s_bs", 1, 2, 1024, 64, block_sparse=True, seed=3)):
        inp = wl.make_inputs(w)
        stride = bench.row_stride(w)
        assert stride == 4
        _, work = bench.oracle_tasks(w, inp, 0, w.B * w.H * stride)
        want = wl.flop_count(w, inp.raw("mask") if w.block_sparse else None) / 1e12
        assert abs(work - want) <= 1e-9 * want, (w.name, work, want)
        tasks, _ = bench.oracle_tasks(w, inp, 0, w.B * w.H * stride)
        rows = sorted(r for t in tasks[:stride * w.B * w.H:w.B * w.H] for r in t[-1])
        assert rows == list(range(w.N))  # the offsets of one head cover every row once
