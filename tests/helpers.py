"""Shared helpers of the parity tests: move seeded inputs to the GPU, run the oracle, compare."""
from __future__ import annotations

import numpy as np
import torch

from exact_attention_fa_gb300 import workloads as wl

# Tolerances (see the module docstrings of the tests for where each comes from).
FP32_MAX_ABS = 1e-5
BF16_O_MAX_ABS = 1e-2
BF16_O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-4
GRAD_REL_FRO = 2e-2


def to_device(inp: wl.Inputs, name: str, device) -> torch.Tensor:
    a = inp.raw(name)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    if a.dtype == np.uint8:
        return torch.from_numpy(a).to(device)
    return torch.from_numpy(a).to(device)


def rel_fro(got: np.ndarray, want: np.ndarray) -> float:
    return float(np.linalg.norm((got - want).ravel()) / max(np.linalg.norm(want.ravel()), 1e-300))


def compare_o(got: np.ndarray, want: np.ndarray, bf16: bool, relative_above_one: bool = False):
    """relative_above_one: entries with |O| > 1 are compared relative to |O| (bf16 keeps 8
    significant bits, so an output of size 3 is already rounded by up to 0.0078 on its own)."""
    err = np.abs(got.astype(np.float64) - want)
    if relative_above_one:
        err = err / np.maximum(1.0, np.abs(want))
    if bf16:
        assert err.max() <= BF16_O_MAX_ABS, f"max abs {err.max():.3e}"
        assert err.mean() <= BF16_O_MEAN_ABS, f"mean abs {err.mean():.3e}"
    else:
        assert err.max() <= FP32_MAX_ABS, f"max abs {err.max():.3e}"
    return float(err.max()), float(err.mean())


def compare_lse(got: np.ndarray, want: np.ndarray, tol=LSE_MAX_ABS):
    got = got.astype(np.float64)
    both_inf = np.isneginf(got) & np.isneginf(want)
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(got - want))
    assert np.all(np.isfinite(err)), "lse: -inf mismatch"
    assert err.max() <= tol, f"lse max abs {err.max():.3e}"
    return float(err.max())
