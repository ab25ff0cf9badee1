"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (a plugin that is handed only its input and output buffers, a serving runtime that
forbids cudaMalloc once it runs) cannot supply fa_bwd's workspace; this entry point uses the
library's static device scratch instead. These tests call it through the C ABI and check that it
gives what fa_bwd gives with a caller-provided workspace, on two calls in a row of different
problems (which reuse the one shared scratch array), and that too large a problem is refused.

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import helpers as H
from exact_attention_fa_gb300 import binding as fa
from exact_attention_fa_gb300 import workloads as wl


def run_pair(w, device):
    inp = wl.make_inputs(w, with_do=True)
    q, k, v, do = (H.to_device(inp, n, device) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_forward(q, k, v, w.softmax_scale, causal=w.causal)
    want = fa.attention_backward(q, k, v, o, lse, do, w.softmax_scale, causal=w.causal)
    dq = torch.full(q.shape, float("nan"), dtype=torch.float32, device=device)
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    fa.fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, w.softmax_scale, w.causal)
    fa.fa_check_device_error()
    return (dq, dk, dv), want


@pytest.mark.gpu
def test_noalloc_matches_workspace_backward_on_two_calls(cuda):
    problems = [wl.Workload("noalloc_a", 2, 4, 1000, 128, causal=True, seed=61),
                wl.Workload("noalloc_b", 1, 8, 640, 64, causal=False, seed=62)]
    for w in problems:
        got, want = run_pair(w, cuda)
        for name, g, r in zip(("dq", "dk", "dv"), got, want):
            g64, r64 = g.double().cpu().numpy(), r.double().cpu().numpy()
            assert np.all(np.isfinite(g64)), name
            err = np.linalg.norm(g64 - r64) / np.linalg.norm(r64)
            assert err <= H.GRAD_REL_FRO, f"{w.name} {name}: {err:.3e}"
        # dK and dV are written once per key tile by the same kernels: identical bits
        assert torch.equal(got[1], want[1]) and torch.equal(got[2], want[2])


def test_noalloc_refuses_problems_beyond_its_scratch(lib_path):
    lib = fa.load(lib_path)
    p = ctypes.c_void_p(0x10000)
    B, Hh, N, d = 8, 32, 8192, 64  # needs 144 MiB of scratch
    assert fa.fa_bwd_workspace_bytes(B, Hh, N, d) > fa.FA_NOALLOC_SCRATCH_BYTES
    st = lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, Hh, N, d, 0.088, 1, None)
    assert st == 8  # FA_ERR_SCRATCH_LIMIT
    assert b"scratch" in lib.fa_status_string(st)
    assert lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, 0, Hh, N, d, 0.088, 1, None) == 1
