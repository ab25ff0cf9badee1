"""The C-ABI library builds, loads and exports every symbol include/fa.h declares (no GPU needed).

Only argument validation runs here: each call below is rejected before anything touches a GPU.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "fa.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(fa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("fa_fwd", "fa_fwd_fp32", "fa_fwd_fp32_fa1", "fa_fwd_blocksparse", "fa_fwd_fp8",
                 "fa_bwd", "fa_bwd_workspace_bytes", "fa_bwd_noalloc",
                 "fa_decode", "fa_decode_ctas", "fa_decode_workspace_bytes",
                 "fa_check_device_error", "fa_status_string", "fa_abi_version"):
        assert want in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_signatures_cover_the_header(lib_path):
    from exact_attention_fa_gb300 import binding
    assert sorted(n for n, _, _ in binding.SIGNATURES) == declared_functions()
    binding.load(lib_path)


@pytest.fixture(scope="module")
def lib(lib_path):
    from exact_attention_fa_gb300 import binding
    return binding.load(lib_path)


P = ctypes.c_void_p


def fake(addr=0x10000):
    return P(addr)


def test_status_strings(lib):
    assert lib.fa_status_string(0) == b"ok"
    assert b"aligned" in lib.fa_status_string(3)
    assert lib.fa_status_string(999) == b"unknown status"
    assert lib.fa_abi_version() >> 16 == 2


@pytest.mark.parametrize("args,want", [
    # null pointer
    ((P(0), fake(), fake(), fake(), fake(), 1, 1, 128, 64, 0.125, 0), 1),
    # bad sizes / scale
    ((fake(), fake(), fake(), fake(), fake(), 0, 1, 128, 64, 0.125, 0), 1),
    ((fake(), fake(), fake(), fake(), fake(), 1, 1, 0, 64, 0.125, 0), 1),
    ((fake(), fake(), fake(), fake(), fake(), 1, 1, 128, 64, 0.0, 0), 1),
    ((fake(), fake(), fake(), fake(), fake(), 1, 1, 128, 64, float("nan"), 0), 1),
    # unsupported head dim
    ((fake(), fake(), fake(), fake(), fake(), 1, 1, 128, 96, 0.125, 0), 2),
    # misaligned
    ((fake(0x10008), fake(), fake(), fake(), fake(), 1, 1, 128, 64, 0.125, 0), 3),
    # too large
    ((fake(), fake(), fake(), fake(), fake(), 1 << 16, 1 << 16, 1024, 64, 0.125, 0), 7),
])
def test_fwd_validation(lib, args, want):
    assert lib.fa_fwd(*args, None) == want


def test_blocksparse_validation(lib):
    base = (fake(), fake(), fake(), fake(), fake(), 1, 1)
    assert lib.fa_fwd_blocksparse(*base, 256, 64, 0.125, 0, P(0), None) == 1  # no mask
    assert lib.fa_fwd_blocksparse(*base, 200, 96, 0.125, 1, fake(), None) == 2  # head dim


def test_decode_validation(lib):
    q = (fake(), fake(), fake(), fake(), fake())
    ws = fake()
    assert lib.fa_decode(P(0), *q[1:], 1, 1, 1, 100, 64, 0.125, 0, ws, None) == 1  # null q
    assert lib.fa_decode(*q, 1, 1, 1, 100, 64, 0.125, 0, P(0), None) == 1  # no workspace
    assert lib.fa_decode(*q, 1, 1, 0, 100, 64, 0.125, 0, ws, None) == 1  # Nq = 0
    assert lib.fa_decode(*q, 1, 1, 1, 0, 64, 0.125, 0, ws, None) == 1  # Nk = 0
    assert lib.fa_decode(*q, 1, 1, 9, 100, 64, 0.125, 0, ws, None) == 2  # Nq > 8
    assert lib.fa_decode(*q, 1, 1, 1, 100, 96, 0.125, 0, ws, None) == 2  # head dim
    assert lib.fa_decode(*q, 1, 1, 1, 100, 64, 0.125, -1, ws, None) == 1  # n_ctas
    assert lib.fa_decode(*q, 1, 1, 1, 100, 64, 0.125, 1025, ws, None) == 1
    assert lib.fa_decode(*q, 1, 1, 1, 100, 64, 0.0, 0, ws, None) == 1  # scale
    assert lib.fa_decode(fake(0x10008), *q[1:], 1, 1, 1, 100, 64, 0.125, 1, ws, None) == 3


def test_decode_workspace_and_ctas(lib):
    # pieces: min(key blocks, 1024) CTAs + B*H heads, Nq rows of d + 1 floats each; blocks of 128
    # keys at d = 128, 256 at d = 64
    assert lib.fa_decode_workspace_bytes(2, 3, 4, 1000, 128) == (6 * 8 + 6) * 4 * 129 * 4
    assert lib.fa_decode_workspace_bytes(2, 3, 4, 1000, 64) == (6 * 4 + 6) * 4 * 65 * 4
    assert lib.fa_decode_workspace_bytes(8, 32, 1, 32768, 128) == (1024 + 256) * 129 * 4
    assert lib.fa_decode_workspace_bytes(1, 1, 9, 100, 64) == 0  # unsupported sizes
    assert lib.fa_decode_ctas(1, 1, 9, 100, 64) == 0


def test_bwd_blocksparse_validation(lib):
    ptrs = [fake()] * 9
    assert lib.fa_bwd_blocksparse(*ptrs, 1, 1, 256, 64, 0.125, 0, P(0), fake(), None) == 1  # mask
    assert lib.fa_bwd_blocksparse(*ptrs, 1, 1, 256, 96, 0.125, 0, fake(), fake(), None) == 2
    # more query tiles than the kernel's bitmask holds (2048 tiles)
    assert lib.fa_bwd_blocksparse(*ptrs, 1, 1, 2049 * 128, 64, 0.125, 0, fake(), fake(), None) == 2


def test_fp32_validation(lib):
    base = (fake(), fake(), fake(), fake(), fake(), 1, 1, 64)
    for fn in (lib.fa_fwd_fp32, lib.fa_fwd_fp32_fa1):
        assert fn(*base, 48, 0.125, 0, None) == 2
        assert fn(*base, 256, 0.125, 0, None) == 2
        assert fn(fake(), fake(), fake(), fake(), P(0), 1, 1, 64, 64, 0.125, 0, None) == 1
        assert fn(fake(), fake(), fake(), fake(), fake(0x10004), 1, 1, 64, 64, 0.125, 0, None) == 3


def test_bwd_validation_and_workspace(lib):
    # per padded row: lse2 and D (fp32), and at d = 64 their two 32-byte bf16 operand rows
    # rows x (8 or 72 bytes), then 4 * (1 + B*H) bytes of counters rounded up to 16
    assert lib.fa_bwd_workspace_bytes(2, 3, 100, 64) == 2 * 3 * 128 * 72 + 32
    assert lib.fa_bwd_workspace_bytes(1, 1, 256, 128) == 256 * 8 + 16
    assert lib.fa_bwd_workspace_bytes(4, 16, 4096, 128) == 64 * 4096 * 8 + 272
    assert lib.fa_bwd_workspace_bytes(0, 3, 100, 64) == 0
    assert lib.fa_bwd_workspace_bytes(1, 1, 256, 96) == 0
    ptrs = [fake()] * 9
    assert lib.fa_bwd(*ptrs, 1, 1, 128, 64, 0.125, 1, P(0), None) == 1
    assert lib.fa_bwd(*ptrs, 1, 1, 128, 80, 0.125, 1, fake(), None) == 2


def test_no_device_here_is_reported_not_crashed(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.fa_fwd(fake(), fake(), fake(), fake(), fake(), 1, 1, 128, 64, 0.125, 0, None) == 6


def test_selftest_validation(lib):
    assert lib.fa_selftest_wait_timeout(0, None) == 1
    assert lib.fa_selftest_wait_timeout(20000001, None) == 1


# (pointers, B, H, N, d, scale) cases that fa_bwd rejects before anything touches a GPU
BAD_BWD_ARGS = [
    ([P(0)] + [fake()] * 8, 1, 1, 128, 64, 0.125),             # null q
    ([fake()] * 8 + [P(0)], 1, 1, 128, 64, 0.125),             # null dv
    ([fake()] * 9, 0, 1, 128, 64, 0.125),                      # B = 0
    ([fake()] * 9, 1, 1, 0, 64, 0.125),                        # N = 0
    ([fake()] * 9, 1, 1, 128, 64, float("nan")),               # scale
    ([fake()] * 9, 1, 1, 128, 96, 0.125),                      # head dim
    ([fake()] * 9, 8, 32, 8192, 96, 0.125),                    # head dim of a large problem
    ([fake(0x10008)] + [fake()] * 8, 1, 1, 128, 64, 0.125),    # misaligned q
    ([fake(0x10008)] + [fake()] * 8, 8, 32, 8192, 64, 0.125),  # misaligned, large problem
    ([P(0)] + [fake()] * 8, 8, 32, 8192, 128, 0.125),          # null q, large problem
    ([fake()] * 9, 1 << 16, 1 << 16, 1024, 64, 0.125),         # too large to index
]


@pytest.mark.parametrize("case", range(len(BAD_BWD_ARGS)))
def test_bwd_noalloc_reports_fa_bwds_status(lib, case):
    """fa_bwd_noalloc runs fa_bwd's argument checks first and in the same order, so a bad
    argument gets the same status from both, whatever the problem's size."""
    ptrs, B, Hh, N, d, scale = BAD_BWD_ARGS[case]
    want = lib.fa_bwd(*ptrs, B, Hh, N, d, scale, 1, fake(), None)
    assert want in (1, 2, 3, 7)
    assert lib.fa_bwd_noalloc(*ptrs, B, Hh, N, d, scale, 1, None) == want


def test_bwd_noalloc_scratch_limit_after_argument_checks(lib):
    ptrs = [fake()] * 9
    # 4 MiB: 58240 padded rows at d = 64 (72 bytes each), 524160 at d = 128 (8 bytes each), plus
    # 16 bytes of counters
    assert lib.fa_bwd_noalloc(*ptrs, 1, 1, 58241, 64, 0.125, 0, None) == 8
    assert lib.fa_bwd_noalloc(*ptrs, 1, 1, 524161, 128, 0.125, 0, None) == 8
    # within the limit the call goes on to the device, which this machine does not have
    import torch
    if not torch.cuda.is_available():
        assert lib.fa_bwd_noalloc(*ptrs, 1, 1, 58240, 64, 0.125, 0, None) == 6
        assert lib.fa_bwd_noalloc(*ptrs, 1, 1, 524160, 128, 0.125, 0, None) == 6


def test_fp8_validation(lib):
    import torch
    base = (fake(), fake(), fake(), fake(), fake(), 1, 1, 256)
    if not torch.cuda.is_available():
        assert lib.fa_fwd_fp8(*base, 128, 0.088, 1.0, 0, None) == 6  # valid: no device here
    assert lib.fa_fwd_fp8(*base, 64, 0.088, 1.0, 0, None) == 2      # d = 128 only
    assert lib.fa_fwd_fp8(*base, 128, 0.088, float("inf"), 0, None) == 1
    assert lib.fa_fwd_fp8(*base, 128, -1.0, 1.0, 0, None) == 1
    assert lib.fa_fwd_fp8(P(0), *base[1:], 128, 0.088, 1.0, 0, None) == 1
    assert lib.fa_fwd_fp8(fake(0x10001), *base[1:], 128, 0.088, 1.0, 0, None) == 3


def test_exp2_emulation_setting(lib):
    assert lib.fa_get_exp2_emulation() == 0  # the default: every exponential on the SFU
    assert lib.fa_set_exp2_emulation(3) == 1 and lib.fa_set_exp2_emulation(-4) == 1
    assert lib.fa_set_exp2_emulation(4) == 0 and lib.fa_get_exp2_emulation() == 4
    assert lib.fa_set_exp2_emulation(0) == 0 and lib.fa_get_exp2_emulation() == 0
