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
    if a.dtype == np.uint8 and name != "mask":  # e4m3 codes
        return torch.from_numpy(a).to(device).view(torch.float8_e4m3fn)
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


# ------------------------------------------------------------------------------ e4m3 forward
# The fp8 forward multiplies e4m3 Q, K, V exactly (fp32 accumulation) and differs from the
# definition on the same e4m3 inputs by one rounding: P is rounded to e4m3 (3 mantissa bits) as
# the A operand of the P V product, while l sums the unrounded fp32 P. Rounding to nearest leaves
# a relative error of at most half an ulp, 2^-4, for normal values and an absolute error of at
# most half the subnormal spacing 2^-9 below 2^-6; treated as independent and uniform over the
# keys, the error of O_ik = sum_j P_j V_jk / l has standard deviation
#     sigma_ik = sqrt(sum_j var_j V_jk^2) / l,   var_j = (2^-4)^2 / 3 * P_j^2 + (2^-10)^2,
# with P_j = exp(S_j - max) (the kernel's P is this times a power of two >= 1 per key tile, which
# only shrinks the subnormal term; the term is taken without the uniform 1/3, conservatively).
# The bf16 output adds a rounding of at most 2^-9 |O|. Bound per element: 6 sigma + 2^-8 |O| +
# 1e-6; and the root mean square of error / sigma_total must stay below 1.5.
FP8_HALF_ULP_REL = 2.0 ** -4
FP8_HALF_SUB = 2.0 ** -10
FP8_Z = 6.0


def fp8_sigma(q, k, v, scale, causal=False, block_mask=None, rows=None):
    """(O reference, sigma) for the rows `rows` of one head: the per-element standard deviation of
    the e4m3 forward's rounding error, by the model above (q, k, v: the exact e4m3 values)."""
    from oracle import attention as orc
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    S = scale * (q[rows] @ k.T)
    ok = orc.allowed_keys(rows, k.shape[0], causal, block_mask)
    S = np.where(ok, S, -np.inf)
    m = S.max(axis=1)
    m = np.where(np.isfinite(m), m, 0.0)
    Pu = np.exp(S - m[:, None])
    ell = Pu.sum(axis=1)
    ell = np.where(ell > 0, ell, 1.0)
    var = FP8_HALF_ULP_REL ** 2 / 3.0 * Pu ** 2 + np.where(ok, FP8_HALF_SUB ** 2, 0.0)
    sigma = np.sqrt(var @ (v ** 2)) / ell[:, None]
    return (Pu @ v) / ell[:, None], sigma


def compare_o_fp8(got, want, sigma):
    """Per-element bound and root-mean-square check of the e4m3 forward's O (see above)."""
    got = got.astype(np.float64)
    err = np.abs(got - want)
    bound = FP8_Z * sigma + 2.0 ** -8 * np.abs(want) + 1e-6
    worst = float((err / bound).max())
    assert worst <= 1.0, f"fp8 O: error {worst:.2f} x its bound"
    s_tot = np.sqrt(sigma ** 2 + (2.0 ** -9 * np.abs(want)) ** 2 / 3.0) + 1e-7
    rms = float(np.sqrt(np.mean((err / s_tot) ** 2)))
    assert rms <= 1.5, f"fp8 O: rms error {rms:.2f} sigma"
    return worst, rms
