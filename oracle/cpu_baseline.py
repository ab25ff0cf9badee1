"""Runs the fp64 oracle on one (b, h) head for the CPU-baseline timing of bench.py.

Test/benchmark infrastructure only (imported by bench.py's cpu_baseline leg and its reference
arm). It holds no arithmetic of its own: it decodes the seeded bf16 inputs and calls the oracle's
forward and backward as they stand.
"""
from __future__ import annotations

import numpy as np

from . import attention as orc


def _f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def warm(_: int) -> int:
    """Touches numpy and the oracle once so that worker start-up is not timed."""
    orc.forward_head(np.ones((2, 2)), np.ones((2, 2)), np.ones((2, 2)), 1.0)
    return 0


def run_head(task) -> float:
    """task = (q, k, v, do bf16 bit arrays [N, d] (do may be None), scale, causal, block_mask).

    Returns the checksum of the outputs (so the work cannot be skipped)."""
    q, k, v, do, scale, causal, block_mask = task
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    O, lse = orc.forward_head(qf, kf, vf, scale, causal=causal, block_mask=block_mask)
    total = float(O.sum())
    if do is not None:
        dq, dk, dv = orc.backward_head(qf, kf, vf, _f64(do), scale, causal=causal,
                                       block_mask=block_mask)
        total += float(dq.sum() + dk.sum() + dv.sum())
    return total
