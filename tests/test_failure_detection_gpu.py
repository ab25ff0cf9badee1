"""Failure detection without a GPU fault: every on-chip wait of the kernels is bounded.

The self-test kernel waits on a barrier that nothing ever arrives at; the wait must give up after
its bound, the device error word must report FA_ERR_DEVICE_TIMEOUT through the C ABI, the word
must be cleared by reading it, and the context must remain usable for the real kernels.
"""
import time

import pytest
import torch

from exact_attention_fa_gb300 import binding as fa

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda):
    fa.fa_check_device_error()  # start clean
    t0 = time.perf_counter()
    fa.fa_selftest_wait_timeout(20000)  # 20 ms bound
    with pytest.raises(fa.FAError) as e:
        fa.fa_check_device_error()
    elapsed = time.perf_counter() - t0
    assert e.value.status == 5  # FA_ERR_DEVICE_TIMEOUT
    assert 0.015 < elapsed < 5.0
    fa.fa_check_device_error()  # the word was cleared by the read
    q = torch.randn(1, 1, 256, 64, device=cuda).bfloat16()
    o, lse = fa.attention_forward(q, q, q)
    fa.fa_check_device_error()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_selftest_rejects_bad_bounds(cuda):
    with pytest.raises(fa.FAError):
        fa.fa_selftest_wait_timeout(0)
