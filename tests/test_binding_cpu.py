"""The Python binding rejects malformed arguments before any library call, and has no fallback:
host tensors are refused rather than computed on the CPU (no GPU needed for these checks)."""
import pytest
import torch

from exact_attention_fa_gb300 import binding as fa


def bf16(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


def test_host_tensors_are_refused_not_computed():
    q = bf16(1, 2, 64, 64)
    with pytest.raises(ValueError, match="CUDA"):
        fa.attention_forward(q, q.clone(), q.clone())
    with pytest.raises(ValueError, match="CUDA"):
        fa.fa_fwd(q, q, q, q.clone(), torch.zeros(1, 2, 64), 0.125)


def test_rank_shape_and_dtype_checks():
    q = bf16(1, 2, 64, 64)
    lse = torch.zeros(1, 2, 64)
    with pytest.raises(ValueError, match=r"\[B, H, N, d\]"):
        fa.fa_fwd(bf16(2, 64, 64), q, q, q, lse, 0.125)
    with pytest.raises(ValueError, match="shape mismatch"):
        fa.fa_fwd(q, bf16(1, 2, 32, 64), q, q, lse, 0.125)
    with pytest.raises(TypeError, match="bfloat16"):
        fa.fa_fwd(q, q.float(), q, q, lse, 0.125)
    with pytest.raises(TypeError, match="float32"):
        fa.fa_fwd_fp32(q, q, q, q, lse, 0.125)
    with pytest.raises(TypeError, match="float32"):
        fa.fa_fwd_fp32_fa1(q.float(), q.float(), q, q.float(), lse, 0.125)


def test_non_contiguous_views_are_refused():
    base = bf16(1, 2, 64, 128)
    view = base[..., :64]  # [1, 2, 64, 64] with a row stride of 128
    assert not view.is_contiguous()
    with pytest.raises(ValueError):
        fa.fa_fwd(view, view, view, view, torch.zeros(1, 2, 64), 0.125)


def test_block_mask_is_bf16_only():
    q = torch.zeros(1, 1, 128, 64)
    with pytest.raises(ValueError, match="bf16 only"):
        fa.attention_forward(q, q, q, block_mask=torch.ones(1, 1, dtype=torch.uint8))


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(fa, "_lib", None)
    with pytest.raises(fa.FAError, match="missing"):
        fa.load(str(tmp_path / "libfa_gb300.so"))


def test_oracle_side_loads_no_product_code():
    """The oracle and the input generator import neither the binding nor the library."""
    import subprocess
    import sys
    code = ("import sys, oracle.cpu_baseline, oracle.attention; "
            "import exact_attention_fa_gb300.workloads; "
            "bad = [m for m in ('exact_attention_fa_gb300.binding', 'exact_attention_fa_gb300.build',"
            " 'torch') if m in sys.modules]; print(bad); assert not bad")
    root = __import__("os").path.dirname(__import__("os").path.dirname(__file__))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


def test_package_exports_resolve_lazily():
    import exact_attention_fa_gb300 as pkg
    assert pkg.fa_fwd is fa.fa_fwd and pkg.fa_fwd_fp8 is fa.fa_fwd_fp8
    with pytest.raises(AttributeError):
        pkg.no_such_entry_point
