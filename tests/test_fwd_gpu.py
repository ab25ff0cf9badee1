"""Forward parity: the CUDA kernels against the fp64 oracle on the same seeded inputs.

Tolerances: fp32 path max-abs 1e-5 on O; bf16 path max-abs 1e-2 and mean-abs 1e-3 on O; lse
max-abs 1e-4 (lse is formed in fp32 from exact bf16 x bf16 products, so its error is a few fp32
ulps of values of size ~10).
"""
import numpy as np
import pytest
import torch

import helpers as H
from exact_attention_fa_gb300 import binding as fa
from exact_attention_fa_gb300 import workloads as wl
from oracle import attention as orc

pytestmark = pytest.mark.gpu


def tile_rows(N, rng):
    """Rows that put a sample in every CTA and every warp of it: in each 128-row query tile one
    random row from each 32-row group (one softmax warp's TMEM lanes), plus the head's first and
    last rows and the rows around the first tile boundary."""
    picks = [np.arange(g, min(g + 32, N)) for g in range(0, N, 32)]
    rows = [rng.choice(p) for p in picks]
    return np.unique(np.concatenate([rows, [0, N - 1, min(N - 1, 127), min(N - 1, 128)]]))


def run_and_compare(w: wl.Workload, device, rows="all", heads=None, relative_above_one=False):
    """Runs the forward of workload w on the GPU and compares it with the oracle on every head
    (or `heads` sampled ones): every row (rows="all") or the tile_rows sample (rows="tiles")."""
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, device) for n in ("q", "k", "v"))
    mask_np = inp.raw("mask") if w.block_sparse else None
    mask = H.to_device(inp, "mask", device) if w.block_sparse else None
    o, lse = fa.attention_forward(q, k, v, w.softmax_scale, causal=w.causal, block_mask=mask)
    fa.fa_check_device_error()
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    rng = np.random.default_rng(1234)
    all_heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    if heads is not None:
        sel = rng.choice(len(all_heads), size=min(heads, len(all_heads)), replace=False)
        all_heads = [all_heads[i] for i in sorted(sel)]
    worst = 0.0
    for b, h in all_heads:
        sel_rows = np.arange(w.N) if rows == "all" else tile_rows(w.N, rng)
        qf, kf, vf = (inp.f64_head(n, b, h) for n in ("q", "k", "v"))
        O_ref, lse_ref = orc.forward_head(qf, kf, vf, w.softmax_scale, causal=w.causal,
                                          block_mask=mask_np, rows=sel_rows)
        mx, _ = H.compare_o(o[b, h, sel_rows], O_ref, bf16=(w.dtype == "bf16"),
                            relative_above_one=relative_above_one)
        H.compare_lse(lse[b, h, sel_rows], lse_ref)
        worst = max(worst, mx)
    return worst, o, lse


# ------------------------------------------------------------------------- fp32 (FMA) path

def test_single_head_fp32_full(cuda):
    w = wl.WORKLOADS["single_head_fp32"]
    worst, _, _ = run_and_compare(w, cuda)
    assert worst < 1e-6  # the toy fp32 kernel of the quant67 page reports 4.12e-7


@pytest.mark.parametrize("N", [1, 31, 257])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_fp32_shapes(cuda, N, d, causal):
    w = wl.Workload("fp32_small", 2, 3, N, d, dtype="fp32", causal=causal, seed=11)
    run_and_compare(w, cuda)


@pytest.mark.parametrize("N,d,causal", [(8192, 128, True), (4096, 64, False)])
def test_fp32_long_sequence(cuda, N, d, causal):
    """The fp32 path at sequence lengths far past the specified one (256 and 128 key blocks of
    32 per row, 8-row CTAs): one row of every 32-row group, the first and last rows, against the
    oracle at the fp32 bar (max-abs 1e-5)."""
    w = wl.Workload("fp32_long", 1, 2, N, d, dtype="fp32", causal=causal, seed=16)
    worst, _, _ = run_and_compare(w, cuda, rows="tiles")
    assert worst < 1e-5


def run_fa1(w: wl.Workload, device):
    """fa_fwd_fp32_fa1 on every row against the oracle's plain definition; dense workloads also
    against the oracle's FA-1 form with the kernel's 32-key blocks."""
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, device) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=device)
    fa.fa_fwd_fp32_fa1(q, k, v, o, lse, w.softmax_scale, w.causal)
    fa.fa_check_device_error()
    o = o.cpu().numpy()
    lse = lse.cpu().numpy()
    qf, kf, vf = inp.f64("q"), inp.f64("k"), inp.f64("v")
    worst = 0.0
    for b in range(w.B):
        for h in range(w.H):
            O_ref, lse_ref = orc.forward_head(qf[b, h], kf[b, h], vf[b, h], w.softmax_scale,
                                              causal=w.causal)
            mx, _ = H.compare_o(o[b, h], O_ref, bf16=False)
            H.compare_lse(lse[b, h], lse_ref)
            worst = max(worst, mx)
            if not w.causal:
                O1, lse1 = orc.forward_fa1_head(qf[b, h], kf[b, h], vf[b, h], w.softmax_scale, 32)
                H.compare_o(o[b, h], O1, bf16=False)
                H.compare_lse(lse[b, h], lse1)
    return worst


@pytest.mark.parametrize("d", [32, 64, 96, 128])
@pytest.mark.parametrize("B,Hh,N", [(1, 1, 700), (2, 16, 300)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp32_rows_per_cta(cuda, d, B, Hh, N, causal):
    """The fp32 kernel takes 8 query rows per CTA, or 2 (4 at d > 64) when a grid of 8-row CTAs
    would leave SMs idle: B1 H1 N700 takes the small form over 22 key blocks, B2 H16 N300 the
    8-row form; every row against the oracle."""
    w = wl.Workload("fp32_rows", B, Hh, N, d, dtype="fp32", causal=causal, seed=14)
    run_and_compare(w, cuda)


@pytest.mark.parametrize("d,N", [(32, 740), (64, 375), (96, 250), (64, 40)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp32_small_problem_kernel(cuda, d, N, causal):
    """Small fp32 problems at d <= 96 stage the whole key range in shared memory and split each
    row's keys over 8 warps, merged with the softmax statistics: these sizes are the largest that
    fit (up to 3 blocks of 32 keys per warp) and one where most warps get no key at all."""
    w = wl.Workload("fp32_smem", 1, 1, N, d, dtype="fp32", causal=causal, seed=15)
    run_and_compare(w, cuda)


def test_single_head_fp32_fa1_form(cuda):
    assert run_fa1(wl.WORKLOADS["single_head_fp32"], cuda) < 1e-6


@pytest.mark.parametrize("N", [1, 31, 257])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_fp32_fa1_form_shapes(cuda, N, d, causal):
    run_fa1(wl.Workload("fp32_fa1", 2, 3, N, d, dtype="fp32", causal=causal, seed=12), cuda)


def test_fp32_fa1_form_large_scores(cuda):
    # scale 1: block maxima differ widely, so both rescale factors of the FA-1 update matter
    run_fa1(wl.Workload("fp32_fa1_big", 1, 2, 300, 64, dtype="fp32", scale=1.0, seed=13), cuda)


# ------------------------------------------------------------------------- bf16 tensor-core path

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 77, 128, 129, 256, 300, 640])
def test_bf16_small(cuda, N, d, causal):
    w = wl.Workload("bf16_small", 2, 3, N, d, causal=causal, seed=21)
    run_and_compare(w, cuda)


def test_bf16_large_scores_exercise_rescaling(cuda):
    # scale 1 with d = 128: scores of std ~11, so the running max moves often and the softmax is
    # nearly one-hot (outputs as large as the values themselves, hence the relative bound)
    w = wl.Workload("bf16_big_scores", 1, 2, 1000, 128, scale=1.0, seed=22)
    run_and_compare(w, cuda, relative_above_one=True)


def test_mha_N2048_d64_full(cuda):
    run_and_compare(wl.WORKLOADS["mha_N2048_d64"], cuda)


def test_causal_N8192_d128_every_cta(cuda):
    """The long-sequence causal workload at full size, in the bench's launch configuration: every
    head, a row of every warp of every query tile (so every CTA of the launch)."""
    run_and_compare(wl.WORKLOADS["causal_N8192_d128"], cuda, rows="tiles")


@pytest.mark.parametrize("N,d,causal", [(131072, 128, True), (65536, 64, False)])
def test_long_sequence_one_row_per_query_tile(cuda, N, d, causal):
    """Sequences 8-16 times longer than the specified workloads (1024 / 512 query tiles, up to
    1024 key tiles per row): one random row of every 128-row query tile, plus the first and last
    rows, against the oracle."""
    w = wl.Workload("long_seq", 1, 1, N, d, causal=causal, seed=74)
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, cuda) for n in ("q", "k", "v"))
    o, lse = fa.attention_forward(q, k, v, w.softmax_scale, causal=causal)
    fa.fa_check_device_error()
    rng = np.random.default_rng(75)
    rows = np.unique(np.concatenate([[0, N - 1], np.arange(0, N, 128) + rng.integers(0, 128, N // 128)]))
    qf, kf, vf = (inp.f64_head(n, 0, 0) for n in ("q", "k", "v"))
    O_ref, lse_ref = orc.forward_head(qf, kf, vf, w.softmax_scale, causal=causal, rows=rows,
                                      row_block=256)
    H.compare_o(o[0, 0].float().cpu().numpy()[rows], O_ref, bf16=True)
    H.compare_lse(lse[0, 0].cpu().numpy()[rows], lse_ref)


@pytest.mark.parametrize("B,Hh,N,d,causal", [
    (1, 9, 8192, 128, True),    # K/V of 8 heads fill the 32 MB head group: groups of 8 + 1
    (3, 11, 2048, 128, False),  # groups of 32 + 1
    (1, 35, 4096, 64, True),    # groups of 32 + 3
])
def test_partial_last_head_group(cuda, B, Hh, N, d, causal):
    """CTAs walk heads in groups whose K/V fit in L2; here the last group is a partial one."""
    w = wl.Workload("partial_group", B, Hh, N, d, causal=causal, seed=71)
    run_and_compare(w, cuda, rows="tiles")


# ------------------------------------------------------------------------- block-sparse

@pytest.mark.parametrize("d", [64, 128])
def test_blocksparse_small_full(cuda, d):
    w = wl.Workload("bs_small", 2, 2, 1024, d, block_sparse=True, seed=31)
    run_and_compare(w, cuda)


@pytest.mark.parametrize("d", [64, 128])
def test_blocksparse_ragged_N(cuda, d):
    # N = 1000: an 8 x 8 tile mask whose last row and column cover 104 keys / queries
    w = wl.Workload("bs_ragged", 1, 2, 1000, d, block_sparse=True, seed=36)
    run_and_compare(w, cuda)


@pytest.mark.parametrize("d,N", [(64, 1024), (128, 1000)])
def test_blocksparse_causal(cuda, d, N):
    w = wl.Workload("bs_causal", 2, 2, N, d, causal=True, block_sparse=True, seed=37)
    run_and_compare(w, cuda)


@pytest.mark.parametrize("d", [64, 128])
def test_all_ones_mask_causal_equals_causal_bitwise(cuda, d):
    w = wl.Workload("bs_ones_causal", 1, 2, 700, d, causal=True, seed=38)
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, cuda) for n in ("q", "k", "v"))
    ones = torch.ones((6, 6), dtype=torch.uint8, device=cuda)
    o1, l1 = fa.attention_forward(q, k, v, w.softmax_scale, causal=True)
    o2, l2 = fa.attention_forward(q, k, v, w.softmax_scale, causal=True, block_mask=ones)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_causal_mask_above_diagonal_only_gives_empty_rows(cuda):
    """Causal + a tile mask that keeps only tiles above the diagonal for query tile 0: its rows
    see no key (O = 0, lse = -inf); query tile 1 keeps its diagonal tile."""
    w = wl.Workload("bs_causal_empty", 1, 1, 256, 128, seed=39)
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, cuda) for n in ("q", "k", "v"))
    m = torch.tensor([[0, 1], [0, 1]], dtype=torch.uint8, device=cuda)
    o, lse = fa.attention_forward(q, k, v, w.softmax_scale, causal=True, block_mask=m)
    assert torch.all(o[:, :, :128] == 0) and torch.all(torch.isneginf(lse[:, :, :128]))
    O_ref, lse_ref = orc.forward_head(inp.f64("q")[0, 0], inp.f64("k")[0, 0], inp.f64("v")[0, 0],
                                      w.softmax_scale, causal=True, block_mask=m.cpu().numpy())
    H.compare_o(o[0, 0].float().cpu().numpy(), O_ref, bf16=True)
    H.compare_lse(lse[0, 0].cpu().numpy(), lse_ref)


def test_blocksparse_N16384_d64_every_cta(cuda):
    run_and_compare(wl.WORKLOADS["blocksparse_N16384_d64"], cuda, rows="tiles")


def test_blocksparse_partial_last_head_group(cuda):
    # N = 16384, d = 64: 8 heads per L2 group, 10 heads -> groups of 8 + 2
    w = wl.Workload("bs_partial_group", 1, 10, 16384, 64, block_sparse=True, seed=72)
    run_and_compare(w, cuda, rows="tiles")


def test_all_ones_mask_equals_dense_bitwise(cuda):
    w = wl.Workload("bs_ones", 1, 2, 512, 64, seed=32)
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, cuda) for n in ("q", "k", "v"))
    ones = torch.ones((4, 4), dtype=torch.uint8, device=cuda)
    o1, l1 = fa.attention_forward(q, k, v, w.softmax_scale)
    o2, l2 = fa.attention_forward(q, k, v, w.softmax_scale, block_mask=ones)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_identity_mask_is_per_tile_attention(cuda):
    w = wl.Workload("bs_eye", 1, 1, 512, 128, seed=33)
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, cuda) for n in ("q", "k", "v"))
    eye = torch.eye(4, dtype=torch.uint8, device=cuda)
    o, lse = fa.attention_forward(q, k, v, w.softmax_scale, block_mask=eye)
    for t in range(4):
        sl = slice(128 * t, 128 * t + 128)
        ot, lt = fa.attention_forward(q[:, :, sl].contiguous(), k[:, :, sl].contiguous(),
                                      v[:, :, sl].contiguous(), w.softmax_scale)
        assert torch.equal(o[:, :, sl], ot) and torch.equal(lse[:, :, sl], lt)


def test_empty_mask_rows_give_zero_and_neg_inf(cuda):
    w = wl.Workload("bs_empty", 1, 1, 256, 64, seed=34)
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, cuda) for n in ("q", "k", "v"))
    m = torch.tensor([[0, 0], [1, 1]], dtype=torch.uint8, device=cuda)
    o, lse = fa.attention_forward(q, k, v, w.softmax_scale, block_mask=m)
    assert torch.all(o[:, :, :128] == 0) and torch.all(torch.isneginf(lse[:, :, :128]))
    O_ref, lse_ref = orc.forward_head(inp.f64("q")[0, 0], inp.f64("k")[0, 0], inp.f64("v")[0, 0],
                                      w.softmax_scale, block_mask=m.cpu().numpy())
    H.compare_o(o[0, 0].float().cpu().numpy(), O_ref, bf16=True)
    H.compare_lse(lse[0, 0].cpu().numpy(), lse_ref)


def test_causal_first_row_is_v0(cuda):
    w = wl.Workload("c_first", 1, 1, 300, 64, causal=True, seed=35)
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, cuda) for n in ("q", "k", "v"))
    o, _ = fa.attention_forward(q, k, v, w.softmax_scale, causal=True)
    assert torch.equal(o[0, 0, 0], v[0, 0, 0])


def test_outputs_do_not_touch_neighbours(cuda):
    """Rows past N are never written (ragged tail): guard rows around the output stay intact."""
    w = wl.Workload("guard", 1, 1, 200, 64, seed=36)
    inp = wl.make_inputs(w)
    q, k, v = (H.to_device(inp, n, cuda) for n in ("q", "k", "v"))
    big = torch.full((1, 1, 400, 64), 7.0, dtype=torch.bfloat16, device=cuda)
    lse_big = torch.full((1, 1, 400), 7.0, dtype=torch.float32, device=cuda)
    o = big[:, :, :200]
    lse = lse_big[:, :, :200]
    fa.fa_fwd(q, k, v, o.contiguous() if not o.is_contiguous() else o, lse, w.softmax_scale)
    torch.cuda.synchronize()
    assert torch.all(big[:, :, 200:] == 7.0) and torch.all(lse_big[:, :, 200:] == 7.0)
