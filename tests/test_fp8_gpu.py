"""The e4m3 forward (fa_fwd_fp8) against the fp64 oracle on the same e4m3 inputs.

The kernel's one rounding beyond the definition is P to e4m3 for the P V product; the bound on O
(tests/helpers.py, fp8_sigma / compare_o_fp8) is derived from that rounding and pinned on the CPU
(test_fp8_tolerance_cpu.py). lse sums the unrounded fp32 P and keeps the bf16 path's bound.
"""
import numpy as np
import pytest
import torch

import helpers as H
from exact_attention_fa_gb300 import binding as fa
from exact_attention_fa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def run_fp8(w, device, rows="all", v_scale=1.0):
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, device) for n in ("q", "k", "v"))
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=device)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=device)
    fa.fa_fwd_fp8(q, k, v, o, lse, w.softmax_scale, v_scale, w.causal)
    fa.fa_check_device_error()
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    rng = np.random.default_rng(99)
    worst = rms_max = 0.0
    from oracle import attention as orc
    for b in range(w.B):
        for h in range(w.H):
            if rows == "all":
                sel = np.arange(w.N)
            else:
                g = [rng.choice(np.arange(s, min(s + 32, w.N))) for s in range(0, w.N, 32)]
                sel = np.unique(np.concatenate([g, [0, w.N - 1]]))
            qf, kf, vf = (inp.f64_head(n, b, h) for n in ("q", "k", "v"))
            want, sigma = H.fp8_sigma(qf, kf, vf, w.softmax_scale, w.causal, rows=sel)
            O_ref, lse_ref = orc.forward_head(qf, kf, vf, w.softmax_scale, causal=w.causal,
                                              rows=sel)
            assert np.allclose(want, O_ref, rtol=0, atol=1e-12)
            wk, rms = H.compare_o_fp8(o[b, h, sel] / v_scale, want, sigma)
            H.compare_lse(lse[b, h, sel], lse_ref)
            worst, rms_max = max(worst, wk), max(rms_max, rms)
    return worst, rms_max


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 77, 128, 129, 300, 640])
def test_fp8_small(cuda, N, causal):
    run_fp8(wl.Workload("fp8_small", 2, 3, N, 128, dtype="e4m3", causal=causal, seed=81), cuda)


def test_fp8_large_scores_exercise_rescaling(cuda):
    # scale 1: scores of std ~11, nearly one-hot rows, frequent moves of the running max
    w = wl.Workload("fp8_big", 1, 2, 1000, 128, dtype="e4m3", scale=1.0, seed=82)
    run_fp8(w, cuda)


def test_fp8_causal_N8192_every_cta(cuda):
    run_fp8(wl.WORKLOADS["causal_N8192_d128_fp8"], cuda, rows="tiles")


def test_fp8_partial_last_head_group(cuda):
    # e4m3 K/V of a head at N = 8192: 2 MiB, 16 heads per 32 MB group; 17 heads -> 16 + 1
    w = wl.Workload("fp8_group", 1, 17, 8192, 128, dtype="e4m3", causal=True, seed=83)
    run_fp8(w, cuda, rows="tiles")


def test_fp8_v_scale_multiplies_o_exactly(cuda):
    w = wl.Workload("fp8_vs", 1, 2, 300, 128, dtype="e4m3", causal=True, seed=84)
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, cuda) for n in ("q", "k", "v"))
    outs = []
    for vs in (1.0, 4.0):
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=cuda)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=cuda)
        fa.fa_fwd_fp8(q, k, v, o, lse, w.softmax_scale, vs, True)
        outs.append((o, lse))
    torch.cuda.synchronize()
    assert torch.equal(outs[1][0], outs[0][0] * 4) and torch.equal(outs[1][1], outs[0][1])


def test_fp8_first_causal_row_is_v0(cuda):
    """Row 0 attends to key 0 only: P = 1 is exact in e4m3, so O_0 = V_0 (as bf16)."""
    w = wl.Workload("fp8_first", 1, 1, 200, 128, dtype="e4m3", causal=True, seed=85)
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, cuda) for n in ("q", "k", "v"))
    o, _ = fa.attention_forward(q, k, v, w.softmax_scale, causal=True)
    assert torch.equal(o[0, 0, 0], v[0, 0, 0].to(torch.bfloat16))
