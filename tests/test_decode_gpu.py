"""Decoding parity: fa_decode (split keys + merge) against the fp64 oracle's plain definition.

A few query rows per head attend to every key of that head ("3 · FlashAttention", 3.6). The
tolerances are the bf16 forward's (O max-abs 1e-2, mean-abs 1e-3; lse 1e-4): the kernel rounds
only the output to bf16, and the chunk merge is exact up to fp32 rounding.
"""
import numpy as np
import pytest
import torch

import helpers as H
from exact_attention_fa_gb300 import binding as fa
from exact_attention_fa_gb300 import workloads as wl
from oracle import attention as orc

pytestmark = pytest.mark.gpu


def run_decode(w, device, n_ctas=0, heads=None):
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, device) for n in ("q", "k", "v"))
    o, lse = fa.attention_decode(q, k, v, w.softmax_scale, n_ctas=n_ctas)
    fa.fa_check_device_error()
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    qf, kf, vf = inp.f64("q"), inp.f64("k"), inp.f64("v")
    pairs = [(b, h) for b in range(w.B) for h in range(w.H)]
    if heads is not None:
        rng = np.random.default_rng(7)
        pairs = [pairs[i] for i in sorted(rng.choice(len(pairs), heads, replace=False))]
    for b, h in pairs:
        O_ref, lse_ref = orc.forward_head(qf[b, h], kf[b, h], vf[b, h], w.softmax_scale)
        H.compare_o(o[b, h], O_ref, bf16=True)
        H.compare_lse(lse[b, h], lse_ref)
    return o, lse


@pytest.mark.parametrize("nq,nk,d,ctas", [
    (1, 1, 64, 0),       # one key
    (1, 77, 128, 0),     # one ragged block per head
    (3, 1000, 64, 1),    # one CTA streams all six heads
    (8, 1000, 128, 7),   # the most query rows; ranges cut heads mid-way
    (2, 4097, 64, 0),    # one key past a 256-key block (its second 128-key row box empty)
    (1, 129, 128, 18),   # one block per CTA
    (5, 300, 128, 1024), # more CTAs asked for than there are blocks (capped)
    (4, 2048, 64, 0),
    (1, 4097, 64, 0),    # a key past a 256-key block boundary
    (1, 1000, 64, 7),
    (1, 129, 64, 1024),  # one block per head: its second row box holds one key
    (2, 200, 64, 0),     # the second row box partly valid
])
def test_decode_small(cuda, nq, nk, d, ctas):
    w = wl.Workload("decode_small", 2, 3, nk, d, nq=nq, seed=40 + nq)
    run_decode(w, cuda, ctas)


@pytest.mark.parametrize("d,nq", [(64, 2), (128, 2), (64, 1), (128, 1)])
def test_decode_long_ranges(cuda, d, nq):
    """Eight CTAs, each streaming dozens of blocks through its ring and across a head boundary
    (ragged last block per head)."""
    w = wl.Workload("decode_long", 2, 4, 16384 + 7, d, nq=nq, seed=50 + d + nq)
    run_decode(w, cuda, 8)


def test_decode_cta_counts_agree(cuda):
    w = wl.Workload("decode_counts", 1, 4, 3000, 128, nq=2, seed=48)
    outs = [run_decode(w, cuda, n)[0] for n in (1, 2, 13, 47, 188)]
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 1e-2


def test_decode_large_scores(cuda):
    # scale 1 with d = 128: a nearly one-hot softmax, so chunks' maxima differ widely
    w = wl.Workload("decode_big", 1, 2, 5000, 128, nq=3, scale=1.0, seed=49)
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, cuda) for n in ("q", "k", "v"))
    o, lse = fa.attention_decode(q, k, v, 1.0, n_ctas=9)
    qf, kf, vf = inp.f64("q"), inp.f64("k"), inp.f64("v")
    for h in range(2):
        O_ref, lse_ref = orc.forward_head(qf[0, h], kf[0, h], vf[0, h], 1.0)
        H.compare_o(o[0, h].float().cpu().numpy(), O_ref, bf16=True, relative_above_one=True)
        H.compare_lse(lse[0, h].cpu().numpy(), lse_ref)


def test_decode_N32768_launch_configuration(cuda):
    """The benchmark's per-head size (32768 keys, d = 128, one query row) with the CTA count
    fa_decode picks for the benchmark's 8 x 32 heads, on 4 heads (so each CTA's range covers
    a fraction of a head, as in the benchmark)."""
    full = wl.WORKLOADS["decode_N32768_d128"]
    n = fa.fa_decode_ctas(full.B, full.H, full.nq, full.N, full.d)
    assert n >= 1
    w = full.with_(B=1, H=4)
    run_decode(w, cuda, n)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_eight_rows_long_cache_every_head(cuda, d):
    """Eight query rows against 32768 keys on 32 heads (the bench's cache length, CTAs cutting
    heads mid-way), every head against the oracle."""
    w = wl.Workload("decode_q8_long", 2, 16, 32768, d, nq=8, seed=56 + d)
    run_decode(w, cuda)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_one_and_eight_rows_agree(cuda, d):
    """The one-row results equal the first row of an eight-row call on the same cache (within the
    bf16 tolerance): the zero-padded query rows do not disturb the others."""
    w8 = wl.Workload("decode_rows8", 1, 4, 5000, d, nq=8, seed=57)
    inp = wl.make_inputs(w8)
    q, k, v = (H.to_device(inp, n, cuda) for n in ("q", "k", "v"))
    o8, l8 = fa.attention_decode(q, k, v, w8.softmax_scale)
    o1, l1 = fa.attention_decode(q[:, :, :1].contiguous(), k, v, w8.softmax_scale)
    torch.cuda.synchronize()
    assert (o1.float() - o8[:, :, :1].float()).abs().max().item() <= H.BF16_O_MAX_ABS
    assert (l1 - l8[:, :, :1]).abs().max().item() <= H.LSE_MAX_ABS
