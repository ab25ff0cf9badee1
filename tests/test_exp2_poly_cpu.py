"""The software exponential's coefficients (csrc/fa_ptx.cuh) are the Remez minimax fit of 2^f on
[-1/2, 1/2] (exact_attention_fa_gb300/exp2_poly_fit.py), and in fp32 they keep the relative error
below 7.5e-5, far under the bf16 rounding of P (2^-9)."""
import os
import re

import numpy as np

from exact_attention_fa_gb300 import exp2_poly_fit as fit

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def kernel_coefficients():
    with open(os.path.join(ROOT, "exact_attention_fa_gb300", "csrc", "fa_ptx.cuh")) as f:
        text = f.read()
    return np.array([float(re.search(rf"kExp2C{i} = ([0-9.e+-]+)f;", text).group(1))
                     for i in range(4)], dtype=np.float32)


def test_kernel_coefficients_are_the_minimax_fit():
    coef, err = fit.remez_exp2(3)
    assert np.array_equal(coef.astype(np.float32), kernel_coefficients())
    assert 7.0e-5 < err < 7.6e-5


def test_fp32_evaluation_error_bound():
    assert fit.fp32_horner_error(kernel_coefficients()) < 7.6e-5 < 2.0 ** -9 / 10


def test_fit_levels_the_error():
    """The minimax property: the error alternates in sign with equal size at degree + 2 points."""
    coef, err = fit.remez_exp2(3)
    g = np.linspace(-0.5, 0.5, 200001)
    e = (np.polyval(coef[::-1], g) - 2.0 ** g) / 2.0 ** g
    segments = np.split(e, np.where(np.diff(np.sign(e)) != 0)[0] + 1)
    peaks = np.array([s[np.argmax(np.abs(s))] for s in segments])
    assert peaks.size == 5  # degree + 2 alternation points
    assert np.all(np.abs(peaks) > 0.999 * err) and np.all(peaks[1:] * peaks[:-1] < 0)
    # a lower-degree fit is much worse (the degree is what buys the accuracy)
    assert fit.remez_exp2(2)[1] > 20 * err
