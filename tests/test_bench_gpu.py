"""bench.py end to end on the GPU: the JSON line carries every key of the reporting contract, for a
forward-only workload, the default forward + backward step and the decoding workload (short
runs)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
        "gpu_launches", "clocks"}


def run_bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.gpu
@pytest.mark.parametrize("workload", ["single_head_fp32", "mha_N2048_d64", "decode_N32768_d128_h8"])
def test_bench_line(cuda, workload):
    args = ["--workload", workload, "--steps", "3", "--warmup", "3", "--no-cpu-baseline"]
    if workload == "mha_N2048_d64":
        args.append("--backward")
    d = run_bench(*args)
    assert KEYS <= set(d), KEYS - set(d)
    assert d["value"] > 0 and d["e2e"]["value"] > 0 and d["gpu_launches"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["roofline"]["peak"] > 0 and 0 < d["roofline"]["frac"]
    assert d["config"]["workload"] == workload
    if workload != "decode_N32768_d128_h8":
        assert 0 < d["ms_per_step_min"] <= d["ms_per_step_median"]
    if workload == "mha_N2048_d64":  # the metric's literal count beside the five contractions
        bwd = d["parts"]["bwd"]
        assert abs(bwd["tflops_at_literal_4BHN2d"] / bwd["tflops"] - 0.4) < 1e-9
    # the fp32 path runs on the FMA pipes; bf16 on the tensor cores, also against the sustained
    # and datasheet peaks; decoding against HBM
    want = {"single_head_fp32": "alu", "mha_N2048_d64": "tensor", "decode_N32768_d128_h8": "hbm"}
    assert d["roofline"]["bound"] == want[workload]
    if want[workload] != "alu":
        assert 0 < d["roofline"]["frac_of_nominal"] < d["roofline"]["frac"]
    if want[workload] == "tensor":
        assert d["roofline"]["frac_of_sustained"] > d["roofline"]["frac"]


@pytest.mark.gpu
def test_bench_decode_reports_bandwidth(cuda):
    d = run_bench("--workload", "decode_N32768_d128_h8", "--steps", "3", "--warmup", "3",
                  "--no-cpu-baseline", "--no-e2e")
    assert d["unit"] == "GB/s" and d["roofline"]["bound"] == "hbm" and d["roofline"]["unit"] == "GB/s"
    assert 0 < d["roofline"]["frac"] < 1.2


@pytest.mark.gpu
def test_bench_default_line_has_per_config_entries(cuda):
    """The default line: the long-sequence causal forward, with one entry per other specified
    workload (CUDA-event ms, TFLOPS, roofline fraction, dominant kernel, clocks, oracle baseline
    for every one of them, the fp32 one included)."""
    d = run_bench("--steps", "3", "--warmup", "3")
    assert KEYS <= set(d), KEYS - set(d)
    assert d["config"]["workload"] == "causal_N8192_d128" and d["config"]["step"] == "forward"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 3 * 8 * 32 * 8192 * 128 * 2
    pc = d["per_config"]
    assert sorted(pc) == sorted(["single_head_fp32", "mha_N2048_d64", "blocksparse_N16384_d64",
                                 "bwd_causal_N4096_d128"])
    for name, e in pc.items():
        assert e["ms_per_step"] > 0 and e["tflops"] > 0, name
        assert 0 < e["roofline"]["frac"] < 1.2 and e["roofline"]["kernel"], name
        assert e["cpu_baseline"]["value"] > 0 and e["cpu_baseline"]["kind"] == "oracle", name
        assert "clocks" in e and e["gpu_launches"] > 0, name
    assert pc["single_head_fp32"]["roofline"]["bound"] == "alu"
    f8 = d["next_rows"]["causal_N8192_d128_fp8"]
    assert f8["config"]["dtype"] == "e4m3" and 0 < f8["roofline"]["frac"] < 1.2
    assert f8["roofline"]["kernel"] == "fwd_pair_kernel<128, true>"
    assert f8["roofline"]["peak"] > 1.9 * d["roofline"]["peak"]  # the fp8 peak
    dec = d["next_rows"]["decode_N32768_d128_q8_b2"]
    assert dec["roofline"]["bound"] == "hbm" and 0 < dec["roofline"]["frac"] < 1.3
    assert dec["gbs"] > 0 and dec["cpu_baseline"]["unit"] == "GB/s"
    for n in ("causal_N8192_d128+exp2_emulation", "mha_N2048_d64+exp2_emulation"):
        e = d["next_rows"][n]
        assert e["exp2_emulation_per32"] == 4 and e["tflops"] > 0 and e["roofline"]["frac"] > 0
    assert pc["bwd_causal_N4096_d128"]["roofline"]["kernel"].startswith("bwd_tc_kernel<128>")
    assert "bwd" in pc["bwd_causal_N4096_d128"]["parts"]
