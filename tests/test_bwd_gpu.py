"""Backward parity: dQ, dK, dV of the CUDA path against the fp64 oracle's softmax calculus.

The GPU backward consumes the GPU forward's O and lse (as a user would); the oracle recomputes
everything from the same bf16 inputs in fp64. Bar: relative Frobenius error <= 2e-2 on each of
dQ, dK, dV.
"""
import numpy as np
import pytest
import torch

import helpers as H
from exact_attention_fa_gb300 import binding as fa
from exact_attention_fa_gb300 import workloads as wl
from oracle import attention as orc

pytestmark = pytest.mark.gpu


def head_errors(got, want):
    """Relative Frobenius error of each gradient of one head. When the oracle's gradient is
    exactly zero (every row of the head has a single allowed key, so dS = 0 and dQ = dK = 0), the
    error is measured against 1% of the head's dV norm instead (a gradient of the same problem
    and scale); everywhere else the denominator is the gradient's own norm."""
    errs = {}
    for n in ("dq", "dk", "dv"):
        den = np.linalg.norm(want[n].ravel())
        if den == 0.0:
            den = 1e-2 * np.linalg.norm(want["dv"].ravel())
        errs[n] = float(np.linalg.norm((got[n] - want[n]).ravel()) / den)
    return errs


def run_bwd(w: wl.Workload, device, heads=None, mask_np=None):
    """Backward of workload w on the GPU against the oracle, head by head (every head, or `heads`
    sampled ones); each head's dQ, dK, dV must meet the bound on its own.
    mask_np: a uint8 tile mask to use instead of the workload's own (block-sparse only)."""
    inp = wl.make_inputs(w, with_do=True)
    q, k, v, do = (H.to_device(inp, n, device) for n in ("q", "k", "v", "do"))
    if w.block_sparse and mask_np is None:
        mask_np = inp.raw("mask")
    mask = torch.from_numpy(mask_np).to(device) if mask_np is not None else None
    o, lse = fa.attention_forward(q, k, v, w.softmax_scale, causal=w.causal, block_mask=mask)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, w.softmax_scale, causal=w.causal,
                                       block_mask=mask)
    fa.fa_check_device_error()
    got = {n: t.float().cpu().numpy() for n, t in (("dq", dq), ("dk", dk), ("dv", dv))}
    for n, t in got.items():
        assert np.all(np.isfinite(t)), f"{n} has non-finite entries"
    all_heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    if heads is not None:
        rng = np.random.default_rng(4321)
        sel = rng.choice(len(all_heads), size=min(heads, len(all_heads)), replace=False)
        all_heads = [all_heads[i] for i in sorted(sel)]
    worst = {"dq": 0.0, "dk": 0.0, "dv": 0.0}
    for b, h in all_heads:
        qf, kf, vf, dof = (inp.f64_head(n, b, h) for n in ("q", "k", "v", "do"))
        gq, gk, gv = orc.backward_head(qf, kf, vf, dof, w.softmax_scale, causal=w.causal,
                                       block_mask=mask_np)
        errs = head_errors({n: got[n][b, h] for n in got}, {"dq": gq, "dk": gk, "dv": gv})
        for n, e in errs.items():
            assert e <= H.GRAD_REL_FRO, f"head ({b}, {h}) {n}: relative Frobenius error {e:.3e}"
            worst[n] = max(worst[n], e)
    return worst


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 64, 128, 200, 384])
def test_bwd_small(cuda, N, d, causal):
    run_bwd(wl.Workload("bwd_small", 2, 2, N, d, causal=causal, seed=41), cuda)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [300, 1024])
def test_bwd_blocksparse_small(cuda, N, d, causal):
    run_bwd(wl.Workload("bwd_bs", 2, 2, N, d, causal=causal, block_sparse=True, seed=44), cuda)


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_blocksparse_unvisited_key_tile(cuda, d):
    """Key tile 1 is in no query tile's mask row: its dK and dV are exactly zero."""
    m = np.array([[1, 0, 0], [1, 0, 0], [1, 0, 1]], np.uint8)
    w = wl.Workload("bwd_bs_empty", 1, 2, 300, d, block_sparse=True, seed=45)
    run_bwd(w, cuda, mask_np=m)
    inp = wl.make_inputs(w, with_do=True)
    q, k, v, do = (H.to_device(inp, n, cuda) for n in ("q", "k", "v", "do"))
    mt = torch.from_numpy(m).to(cuda)
    o, lse = fa.attention_forward(q, k, v, w.softmax_scale, block_mask=mt)
    _, dk, dv = fa.attention_backward(q, k, v, o, lse, do, w.softmax_scale, block_mask=mt)
    assert torch.all(dk[:, :, 128:256] == 0) and torch.all(dv[:, :, 128:256] == 0)


def test_bwd_blocksparse_N4096_d64_sampled(cuda):
    w = wl.Workload("bwd_bs_4096", 1, 8, 4096, 64, block_sparse=True, seed=46)
    run_bwd(w, cuda, heads=2)


def test_bwd_big_scores(cuda):
    run_bwd(wl.Workload("bwd_big", 1, 2, 640, 128, causal=True, scale=0.5, seed=42), cuda)


def test_bwd_mha_N2048_d64_sampled(cuda):
    w = wl.WORKLOADS["mha_N2048_d64"]
    run_bwd(w.with_(backward=True), cuda, heads=4)


def test_bwd_causal_N4096_d128_every_head(cuda):
    """The specified backward workload at full size: all 64 heads, each against the bound."""
    run_bwd(wl.WORKLOADS["bwd_causal_N4096_d128"], cuda)


@pytest.mark.parametrize("N,d,causal", [(32768, 128, True), (16384, 64, False)])
def test_bwd_long_sequence_sampled(cuda, N, d, causal):
    """Sequences 4-8 times longer than the specified backward workload (up to 256 key tiles add
    into a dQ row): dQ at one random row of every query tile and dK, dV at one random key of
    every key tile (plus the first and last), against the oracle's row-blocked backward."""
    w = wl.Workload("bwd_long_seq", 1, 1, N, d, causal=causal, seed=76)
    inp = wl.make_inputs(w, with_do=True)
    q, k, v, do = (H.to_device(inp, n, cuda) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_forward(q, k, v, w.softmax_scale, causal=causal)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, w.softmax_scale, causal=causal)
    fa.fa_check_device_error()
    rng = np.random.default_rng(77)
    pick = lambda: np.unique(np.concatenate([[0, N - 1], np.arange(0, N, 128) + rng.integers(0, 128, N // 128)]))
    rows, cols = pick(), pick()
    qf, kf, vf, dof = (inp.f64_head(n, 0, 0) for n in ("q", "k", "v", "do"))
    gq, gk, gv = orc.backward_head_sampled(qf, kf, vf, dof, w.softmax_scale, rows, cols,
                                           causal=causal)
    got = {"dq": dq[0, 0].float().cpu().numpy()[rows], "dk": dk[0, 0].float().cpu().numpy()[cols],
           "dv": dv[0, 0].float().cpu().numpy()[cols]}
    for n, t in got.items():
        assert np.all(np.isfinite(t)), f"{n} has non-finite entries"
    errs = head_errors(got, {"dq": gq, "dk": gk, "dv": gv})
    for n, e in errs.items():
        assert e <= H.GRAD_REL_FRO, f"{n}: relative Frobenius error {e:.3e}"


@pytest.mark.parametrize("B,Hh,N,d,causal", [
    (1, 17, 2048, 128, True),   # the backward groups heads whose Q, K, V, dO fit in 32 MB: 16 + 1
    (1, 33, 2048, 64, False),   # 32 + 1
])
def test_bwd_partial_last_head_group(cuda, B, Hh, N, d, causal):
    run_bwd(wl.Workload("bwd_partial_group", B, Hh, N, d, causal=causal, seed=73), cuda)


def test_bwd_repeatable_within_tolerance(cuda):
    """dQ is accumulated with floating-point reductions (order may vary between runs); dK and dV
    are written once per key tile and must repeat bit for bit."""
    w = wl.Workload("bwd_rep", 1, 2, 512, 64, causal=True, seed=43)
    inp = wl.make_inputs(w, with_do=True)
    q, k, v, do = (H.to_device(inp, n, cuda) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_forward(q, k, v, w.softmax_scale, causal=True)
    a = fa.attention_backward(q, k, v, o, lse, do, w.softmax_scale, causal=True)
    b = fa.attention_backward(q, k, v, o, lse, do, w.softmax_scale, causal=True)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert torch.allclose(a[0], b[0], rtol=0, atol=1e-5)


@pytest.mark.parametrize("d,N,Hh,sparse", [
    (128, 4096, 10, False),  # causal; heads in groups of 8: 8 + 2
    (128, 4096, 10, True),
    (64, 2048, 40, True),    # groups of 32: 32 + 8
])
def test_bwd_zeroes_dq_whatever_the_buffers_held(cuda, d, N, Hh, sparse):
    """The backward zeroes dQ itself (the first head group's rows in the prep kernel, each later
    group's rows in the main kernel, by the CTAs of the group before) and resets its work
    counters: with dq, dk, dv full of NaN and the workspace full of 0xff bytes beforehand, the
    result is that of fresh buffers, and a query tile that visits no key tile gets dQ = 0."""
    T = (N + 127) // 128
    m = np.ones((T, T), np.uint8)
    m[1, :] = 0  # query tile 1 visits no key tile
    w = wl.Workload("bwd_garbage", 1, Hh, N, d, causal=not sparse, block_sparse=sparse, seed=74)
    inp = wl.make_inputs(w, with_do=True)
    q, k, v, do = (H.to_device(inp, n, cuda) for n in ("q", "k", "v", "do"))
    mt = torch.from_numpy(m).to(cuda) if sparse else None
    o, lse = fa.attention_forward(q, k, v, w.softmax_scale, causal=w.causal, block_mask=mt)
    ref = fa.attention_backward(q, k, v, o, lse, do, w.softmax_scale, causal=w.causal,
                                block_mask=mt)
    dq = torch.full(q.shape, float("nan"), dtype=torch.float32, device=cuda)
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    ws = torch.full((max(16, fa.fa_bwd_workspace_bytes(1, Hh, N, d)),), 255, dtype=torch.uint8,
                    device=cuda)
    if sparse:
        fa.fa_bwd_blocksparse(q, k, v, o, do, lse, dq, dk, dv, w.softmax_scale, False, mt, ws)
    else:
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, w.softmax_scale, True, ws)
    fa.fa_check_device_error()
    assert torch.all(torch.isfinite(dq))
    if sparse:
        assert torch.all(dq[:, :, 128:256] == 0)
    err = (torch.linalg.vector_norm(dq - ref[0]) / torch.linalg.vector_norm(ref[0])).item()
    assert err <= 1e-5, err
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
