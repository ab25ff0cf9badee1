"""The bf16 forward with part of its exponentials computed in software on the FMA pipes
(fa_set_exp2_emulation(4): 4 of every 32 per row, the FA4 idea of "3 · FlashAttention", 3.5),
against the fp64 oracle within the bf16 tolerances, and different from the SFU path (so the
polynomial path is the one that ran)."""
import numpy as np
import pytest
import torch

import helpers as H
from exact_attention_fa_gb300 import binding as fa
from exact_attention_fa_gb300 import workloads as wl
from test_fwd_gpu import run_and_compare

pytestmark = pytest.mark.gpu


@pytest.fixture
def emulation(cuda):
    fa.fa_set_exp2_emulation(4)
    yield
    fa.fa_set_exp2_emulation(0)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 300, 640])
def test_emulated_exp2_small(emulation, cuda, N, d, causal):
    run_and_compare(wl.Workload("poly_small", 2, 3, N, d, causal=causal, seed=91), cuda)


def test_emulated_exp2_large_scores(emulation, cuda):
    w = wl.Workload("poly_big", 1, 2, 1000, 128, scale=1.0, seed=92)
    run_and_compare(w, cuda, relative_above_one=True)


@pytest.mark.parametrize("d", [64, 128])
def test_emulated_exp2_blocksparse_causal(emulation, cuda, d):
    run_and_compare(wl.Workload("poly_bs", 2, 2, 1000, d, causal=True, block_sparse=True,
                                seed=93), cuda)


def test_emulated_exp2_long_sequence_every_cta(emulation, cuda):
    run_and_compare(wl.Workload("poly_long", 1, 9, 8192, 128, causal=True, seed=94), cuda,
                    rows="tiles")


def test_emulated_exp2_runs_its_own_path(cuda):
    w = wl.Workload("poly_diff", 2, 4, 1024, 64, seed=95)
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, cuda) for n in ("q", "k", "v"))
    o_sfu, l_sfu = fa.attention_forward(q, k, v, w.softmax_scale)
    fa.fa_set_exp2_emulation(4)
    try:
        o_poly, l_poly = fa.attention_forward(q, k, v, w.softmax_scale)
    finally:
        fa.fa_set_exp2_emulation(0)
    torch.cuda.synchronize()
    assert fa.fa_get_exp2_emulation() == 0
    assert not torch.equal(l_sfu, l_poly)  # different rounding of some exponentials
    diff = (o_sfu.float() - o_poly.float()).abs().max().item()
    assert 0 < diff <= 2 * H.BF16_O_MAX_ABS
