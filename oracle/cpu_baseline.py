"""Runs the fp64 oracle on one (b, h) head for the CPU-baseline timing of bench.py.

Test/benchmark infrastructure only (imported by bench.py's cpu_baseline leg and its reference
arm). It holds no arithmetic of its own: it decodes the seeded inputs (bf16 bit patterns, e4m3
codes or fp32) and calls the oracle's forward and backward as they stand.
"""
from __future__ import annotations

import numpy as np

from . import attention as orc


def _f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:  # bf16 bit patterns
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if a.dtype == np.uint8:  # e4m3 codes, decoded by the input generator's table
        from exact_attention_fa_gb300.workloads import e4m3_bits_to_f64
        return e4m3_bits_to_f64(a)
    return a.astype(np.float64)


def warm(_: int) -> int:
    """Touches numpy and the oracle once so that worker start-up is not timed."""
    orc.forward_head(np.ones((2, 2)), np.ones((2, 2)), np.ones((2, 2)), 1.0)
    return 0


def run_head(task) -> float:
    """task = (q, k, v, do [N, d] arrays (bf16 bits or fp32; do may be None), scale, causal,
    block_mask, rows). rows: the query rows to compute (None: all of them); the forward of a row
    subset is the same computation restricted to those rows. The backward always takes the whole
    head.

    Returns the checksum of the outputs (so the work cannot be skipped)."""
    q, k, v, do, scale, causal, block_mask, rows = task
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    O, lse = orc.forward_head(qf, kf, vf, scale, causal=causal, block_mask=block_mask, rows=rows)
    total = float(O.sum())
    if do is not None:
        dq, dk, dv = orc.backward_head(qf, kf, vf, _f64(do), scale, causal=causal,
                                       block_mask=block_mask)
        total += float(dq.sum() + dk.sum() + dv.sum())
    return total
