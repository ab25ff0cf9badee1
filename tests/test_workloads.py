"""The seeded input generator (shared by both sides of every parity test)."""
import numpy as np
import torch

from exact_attention_fa_gb300 import workloads as wl


def test_bf16_rounding_matches_torch_round_to_nearest_even():
    x = wl.normal_f32((4096,), seed=7, stream=1) * np.float32(3.7)
    # include exact ties: values halfway between two bf16 numbers
    ties = (np.arange(1, 65, dtype=np.uint32) << np.uint32(16)) | np.uint32(0x8000)
    x = np.concatenate([x, ties.view(np.float32), -ties.view(np.float32)])
    ours = wl.bf16_bits_from_f32(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)
    back = wl.bf16_bits_to_f64(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def test_generator_is_seeded_and_streams_differ():
    a = wl.normal_f32((8, 8), 3, wl.STREAM_Q)
    b = wl.normal_f32((8, 8), 3, wl.STREAM_Q)
    c = wl.normal_f32((8, 8), 3, wl.STREAM_K)
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_block_mask_density_and_diagonal():
    m = wl.block_mask(128, seed=4)
    assert m.dtype == np.uint8 and m.shape == (128, 128)
    assert np.all(np.diag(m) == 1)
    off = m[~np.eye(128, dtype=bool)]
    assert abs(off.mean() - 0.25) < 0.02


def test_flop_counts():
    w = wl.WORKLOADS["mha_N2048_d64"]
    assert wl.flop_count(w) == 4.0 * 4 * 16 * 2048 * 2048 * 64
    wc = wl.WORKLOADS["causal_N8192_d128"]
    assert wl.flop_count(wc) == 2.0 * 8 * 32 * 8192 * 8192 * 128
    assert wl.flop_count(wc, part="bwd") == 2.5 * wl.flop_count(wc)
    wb = wl.WORKLOADS["blocksparse_N16384_d64"]
    mask = wl.block_mask(128, wb.seed)
    assert wl.flop_count(wb, mask) == 4.0 * 2 * 16 * 64 * 128 * 128 * mask.sum()


def test_make_inputs_shapes():
    w = wl.WORKLOADS["mha_N2048_d64"].with_(B=1, H=2, N=130)
    inp = wl.make_inputs(w, with_do=True)
    assert inp.raw("q").shape == (1, 2, 130, 64) and inp.raw("q").dtype == np.uint16
    assert "do" in inp.arrays
    w32 = wl.WORKLOADS["single_head_fp32"]
    inp32 = wl.make_inputs(w32)
    assert inp32.raw("k").dtype == np.float32 and inp32.f64("k").dtype == np.float64


def test_e4m3_table_follows_the_format_definition():
    v = wl.E4M3_VALUES
    assert v[0x00] == 0.0 and v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9  # subnormals
    assert v[0x08] == 2.0 ** -6 and v[0x38] == 1.0 and v[0x7E] == 448.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and v[0xB8] == -1.0
    assert np.all(np.diff(v[:0x7F]) > 0)


def test_e4m3_rounding_matches_torch_round_to_nearest_even():
    x = wl.normal_f32((50000,), seed=8, stream=1) * np.float32(5.0)
    mids = (wl.E4M3_VALUES[1:0x7E] + wl.E4M3_VALUES[2:0x7F]) / 2  # exact ties
    x = np.concatenate([x, mids, -mids, wl.E4M3_VALUES[:0x7F], [2.0 ** -10, 3 * 2.0 ** -11]])
    ours = wl.e4m3_bits_from_f32(x)
    theirs = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(ours, theirs.numpy())
    assert np.all(wl.e4m3_bits_from_f32(np.array([500.0, -1e4])) == [0x7E, 0xFE])  # saturates


def test_e4m3_inputs_decode_exactly():
    w = wl.Workload("f8", 1, 2, 100, 128, dtype="e4m3", seed=3)
    inp = wl.make_inputs(w)
    assert inp.raw("q").dtype == np.uint8
    x = wl.normal_f32((1, 2, 100, 128), 3, wl.STREAM_Q)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(inp.f64("q"), want)
    assert np.array_equal(inp.f64_head("q", 0, 1), want[0, 1])


def test_e4m3_fast_rounding_equals_the_table_search():
    """The integer-arithmetic rounding used for large inputs equals the table search."""
    x = np.concatenate([wl.normal_f32((200000,), 1, 1) * np.float32(s)
                        for s in (0.001, 0.02, 1.0, 30.0, 200.0)])
    mids = (wl.E4M3_VALUES[1:0x7E] + wl.E4M3_VALUES[2:0x7F]) / 2
    x = np.concatenate([x, mids, -mids, wl.E4M3_VALUES[:0x7F],
                        [500.0, -1e4, 448.0, 464.0, 463.9, 2.0 ** -10, -2.0 ** -10, 0.0, -0.0]])
    x = x.astype(np.float32)
    assert np.array_equal(wl.e4m3_bits_from_f32_fast(x), wl.e4m3_bits_from_f32(x))
