"""The e4m3 forward's tolerance (tests/helpers.py, fp8_sigma and compare_o_fp8) against the
rounding it describes, on the CPU: the oracle on e4m3-rounded inputs, with P rounded to e4m3 the
way the kernel rounds it (per 128-key tile against a reference max up to 8 log2 units below the
row's running max), stays within the bound; rounding P to fewer bits, or an error of the size of O
itself, does not."""
import numpy as np
import pytest

import helpers as H
from exact_attention_fa_gb300 import workloads as wl
from oracle import attention as orc


def round_to_bits(x, mant_bits):
    """Round to nearest with `mant_bits` mantissa bits and the e4m3 exponent range (subnormals
    below 2^-6); mant_bits = 3 is e4m3 itself."""
    if mant_bits == 3:
        return wl.e4m3_bits_to_f64(wl.e4m3_bits_from_f32(x))
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -6)))
    q = 2.0 ** (e - mant_bits)
    return np.round(x / q) * q


def emulate_fp8(q, k, v, scale, causal, rng, mant_bits=3):
    """O with P rounded to `mant_bits`: each row's P of key tile j is exp(S - max) times 2^u_j,
    u_j in [0, 8] (the kernel's reference max can sit up to 8 below the running max)."""
    n, N = q.shape[0], k.shape[0]
    rows = np.arange(n)
    S = scale * (q @ k.T)
    ok = orc.allowed_keys(rows, N, causal)
    S = np.where(ok, S, -np.inf)
    m = S.max(axis=1)
    Pu = np.exp(S - m[:, None])
    ell = Pu.sum(axis=1)
    c = 2.0 ** rng.uniform(0, 8, size=(n, -(-N // 128)))
    c = np.repeat(c, 128, axis=1)[:, :N]
    Pq = round_to_bits((Pu * c).astype(np.float32), mant_bits) / c
    return (Pq @ v) / ell[:, None]


def e4m3_head(N, d, seed):
    w = wl.Workload("f8cpu", 1, 1, N, d, dtype="e4m3", seed=seed)
    inp = wl.make_inputs(w)
    return inp.f64("q")[0, 0], inp.f64("k")[0, 0], inp.f64("v")[0, 0], w.softmax_scale


@pytest.mark.parametrize("N,causal", [(300, True), (1000, False), (2048, True)])
def test_fp8_rounding_of_p_stays_within_the_bound(N, causal):
    q, k, v, scale = e4m3_head(N, 128, seed=N)
    rng = np.random.default_rng(N)
    want, sigma = H.fp8_sigma(q, k, v, scale, causal)
    O_ref, _ = orc.forward_head(q, k, v, scale, causal=causal)
    assert np.allclose(want, O_ref, rtol=0, atol=1e-12)  # the model's O is the definition's
    got = emulate_fp8(q, k, v, scale, causal, rng)
    got = wl.bf16_bits_to_f64(wl.bf16_bits_from_f32(got.astype(np.float32)))  # bf16 output
    worst, rms = H.compare_o_fp8(got, want, sigma)
    assert rms > 0.05  # the rounding is visible to the check, not hidden under its floor


@pytest.mark.parametrize("N,causal", [(1000, False), (2048, True)])
def test_fp8_bound_rejects_coarser_rounding(N, causal):
    """P rounded to 1 mantissa bit instead of 3: four times the error, caught."""
    q, k, v, scale = e4m3_head(N, 128, seed=N + 1)
    rng = np.random.default_rng(N)
    want, sigma = H.fp8_sigma(q, k, v, scale, causal)
    got = emulate_fp8(q, k, v, scale, causal, rng, mant_bits=1)
    with pytest.raises(AssertionError):
        H.compare_o_fp8(got, want, sigma)


def test_fp8_bound_rejects_a_misplaced_key_tile():
    """Values of the wrong key tile for one tile of keys (an indexing mistake): caught."""
    q, k, v, scale = e4m3_head(1024, 128, seed=5)
    want, sigma = H.fp8_sigma(q, k, v, scale, False)
    v_bad = v.copy()
    v_bad[256:384] = v[384:512]
    got, _ = orc.forward_head(q, k, v_bad, scale)
    with pytest.raises(AssertionError):
        H.compare_o_fp8(got, want, sigma)
