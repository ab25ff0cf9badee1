"""Pins of the fp64 oracle against things other than itself (CPU only).

* the worked examples the FlashAttention-2 walk-through prints (tests/golden/llmse_worked_examples.json);
* scipy's softmax / logsumexp (K = I, V = I turns attention into a plain row softmax);
* invariants of the definition (convex combination, uniform scores, permutation, N = 1, masks);
* the online recurrence (FA2 deferred normalisation and the FA1 per-block form) for any block size;
* central finite differences and softmax-Jacobian invariants for the backward.
"""
import json
import os

import numpy as np
import pytest
import scipy.special

from oracle import attention as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "llmse_worked_examples.json")
PRINTED_TOL = 0.5e-3 + 1e-9  # the page rounds to 3 decimals


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def scores_as_attention(scores):
    """One query, d = 1: q = [1], k_j = [s_j], scale 1 gives exactly the score row s."""
    s = np.asarray(scores, dtype=np.float64)
    return np.ones((1, 1)), s[:, None]


# ------------------------------------------------------------------ worked examples (printed values)

def test_figure1_deferred_normalisation(golden):
    g = golden["figure1_deferred_normalisation"]
    q, k = scores_as_attention(g["scores"])
    v = np.asarray(g["values"], dtype=np.float64)
    O, lse = orc.forward_head(q, k, v, 1.0)
    assert np.allclose(O[0], g["output"], atol=PRINTED_TOL)
    trace = []
    O2, _ = orc.forward_online_head(q, k, v, 1.0, block=2, trace=trace)
    m, ell, a = trace[-1]
    assert m[0] == 2.0
    assert abs(ell[0] - g["sum_l"]) < PRINTED_TOL
    assert np.allclose(a[0], g["unnormalised_a"], atol=PRINTED_TOL)
    assert np.allclose(O2[0], g["output"], atol=PRINTED_TOL)
    # the row's probabilities: with V = I the output is the probability row itself
    P, _ = orc.forward_head(q, k, np.eye(2), 1.0)
    assert np.allclose(P[0], g["probabilities"], atol=PRINTED_TOL)
    # lse = m + ln l
    assert abs(lse[0] - (2.0 + np.log(g["sum_l"]))) < 1e-3


def test_figure2_chunked_states(golden):
    g = golden["figure2_chunked_update"]
    q, k = scores_as_attention(g["scores"])
    v = np.asarray(g["values"], dtype=np.float64)
    trace = []
    O, lse = orc.forward_online_head(q, k, v, 1.0, block=g["chunk"], trace=trace)
    assert len(trace) == len(g["states_after_each_chunk"])
    for (m, ell, a), want in zip(trace, g["states_after_each_chunk"]):
        assert m[0] == want["m"]
        assert abs(ell[0] - want["l"]) < PRINTED_TOL
        assert np.allclose(a[0], want["a"], atol=PRINTED_TOL)
    # the correction applied at the third chunk: alpha = exp(2 - 3) rescales l and a
    m2, l2, a2 = trace[1]
    alpha = np.exp(m2[0] - trace[2][0][0])
    assert abs(alpha - g["chunk3_correction_factor"]) < PRINTED_TOL
    assert abs(alpha * l2[0] - g["chunk3_corrected_l"]) < PRINTED_TOL
    assert np.allclose(alpha * a2[0], g["chunk3_corrected_a"], atol=PRINTED_TOL)
    assert np.allclose(O[0], g["output"], atol=PRINTED_TOL)
    O_def, lse_def = orc.forward_head(q, k, v, 1.0)
    assert np.allclose(O_def, O, atol=1e-14, rtol=0)
    assert abs(lse_def[0] - lse[0]) < 1e-14


def test_figure3_tile_walkthrough(golden):
    g = golden["figure3_tile_walkthrough"]
    Q = np.asarray(g["Q"], dtype=np.float64)
    K = np.asarray(g["K"], dtype=np.float64)
    V = np.asarray(g["V"], dtype=np.float64)
    S = Q @ K.T
    assert np.array_equal(S[:, :2], g["tile1_scores"])
    assert np.array_equal(S[:, 2:], g["tile2_scores"])
    trace = []
    O, _ = orc.forward_online_head(Q, K, V, 1.0, block=g["tile"], trace=trace)
    # after the first tile both rows have max 2
    assert np.allclose(trace[0][2], g["tile1_a"], atol=PRINTED_TOL)
    m, ell, a = trace[-1]
    assert np.allclose(ell, g["final_l"], atol=PRINTED_TOL)
    assert np.allclose(a, g["final_a"], atol=PRINTED_TOL)
    assert np.allclose(O, g["output"], atol=PRINTED_TOL)
    O_def, _ = orc.forward_head(Q, K, V, 1.0)
    assert np.allclose(O_def, g["output"], atol=PRINTED_TOL)


# ------------------------------------------------------------------ library special cases

def test_softmax_and_logsumexp_match_scipy():
    rng = np.random.default_rng(0)
    X = rng.standard_normal((37, 53)) * 4
    # K = I (d = number of keys), V = I, scale = 1: O is softmax(X) and lse is logsumexp(X)
    O, lse = orc.forward_head(X, np.eye(53), np.eye(53), 1.0)
    assert np.allclose(O, scipy.special.softmax(X, axis=1), atol=1e-15, rtol=1e-12)
    assert np.allclose(lse, scipy.special.logsumexp(X, axis=1), atol=1e-13)
    V = rng.standard_normal((53, 7))
    O2, _ = orc.forward_head(X, np.eye(53), V, 1.0)
    assert np.allclose(O2, scipy.special.softmax(X, axis=1) @ V, atol=1e-13)


def test_scale_multiplies_scores():
    rng = np.random.default_rng(1)
    X = rng.standard_normal((9, 11))
    O, lse = orc.forward_head(X, np.eye(11), np.eye(11), 0.3)
    assert np.allclose(O, scipy.special.softmax(0.3 * X, axis=1), atol=1e-14)
    assert np.allclose(lse, scipy.special.logsumexp(0.3 * X, axis=1), atol=1e-13)


def test_causal_matches_masked_scipy_softmax():
    rng = np.random.default_rng(2)
    n = 19
    X = rng.standard_normal((n, n)) * 3
    O, lse = orc.forward_head(X, np.eye(n), np.eye(n), 1.0, causal=True)
    Xm = np.where(np.tril(np.ones((n, n), dtype=bool)), X, -np.inf)
    assert np.allclose(O, scipy.special.softmax(Xm, axis=1), atol=1e-14)
    assert np.allclose(lse, scipy.special.logsumexp(Xm, axis=1), atol=1e-13)
    assert np.all(np.triu(O, 1) == 0.0)


def test_block_mask_matches_masked_scipy_softmax():
    rng = np.random.default_rng(3)
    tile, nt = 4, 5
    n = tile * nt
    X = rng.standard_normal((n, n)) * 2
    bm = (rng.random((nt, nt)) < 0.4).astype(np.uint8)
    np.fill_diagonal(bm, 1)
    O, lse = orc.forward_head(X, np.eye(n), np.eye(n), 1.0, block_mask=bm, tile=tile)
    full = np.kron(bm, np.ones((tile, tile))).astype(bool)
    Xm = np.where(full, X, -np.inf)
    assert np.allclose(O, scipy.special.softmax(Xm, axis=1), atol=1e-14)
    assert np.allclose(lse, scipy.special.logsumexp(Xm, axis=1), atol=1e-13)


def test_causal_block_mask_ragged_matches_brute_force():
    """Causal and tile masks combined, n not a multiple of the tile: the allowed set is the
    elementwise AND, written out here with plain loops; a query tile whose only tiles lie above
    the diagonal has rows with no key (O = 0, lse = -inf)."""
    rng = np.random.default_rng(4)
    tile, n = 4, 18  # 5 x 5 tile mask, last tile holds 2 keys / queries
    nt = -(-n // tile)
    X = rng.standard_normal((n, n)) * 2
    bm = (rng.random((nt, nt)) < 0.5).astype(np.uint8)
    np.fill_diagonal(bm, 1)
    bm[0, 0] = 0  # rows 0..3 keep only tiles above the diagonal -> empty under causal
    ok = np.zeros((n, n), dtype=bool)
    for i in range(n):
        for j in range(n):
            ok[i, j] = j <= i and bm[i // tile][j // tile] == 1
    O, lse = orc.forward_head(X, np.eye(n), np.eye(n), 1.0, causal=True, block_mask=bm, tile=tile)
    empty = ~ok.any(axis=1)
    assert empty[:4].all() and not empty[4:].any()
    assert np.all(O[empty] == 0.0) and np.all(np.isneginf(lse[empty]))
    Xm = np.where(ok, X, -np.inf)[~empty]
    assert np.allclose(O[~empty], scipy.special.softmax(Xm, axis=1), atol=1e-14)
    assert np.allclose(lse[~empty], scipy.special.logsumexp(Xm, axis=1), atol=1e-13)


@pytest.mark.parametrize("n_q,n_k,splits", [(1, 1, 1), (1, 200, 1), (3, 200, 7), (8, 1000, 13),
                                              (2, 5, 9), (1, 129, 128)])
def test_decode_split_merge_equals_definition(n_q, n_k, splits):
    """Chunked decoding merged by the statistics formula is the plain softmax over all keys
    (closed form, any chunk count, empty chunks included)."""
    q, k, v = rand_head(max(n_q, n_k), 16, 11 + n_k)
    q = q[:n_q] * 2.0
    k, v = k[:n_k], v[:n_k]
    O, lse = orc.decode_split_head(q, k, v, 0.7, splits)
    O_ref, lse_ref = orc.forward_head(q, k, v, 0.7)
    assert np.allclose(O, O_ref, atol=1e-13) and np.allclose(lse, lse_ref, atol=1e-12)


def test_decode_single_key_and_uniform_scores():
    """One key: O = v_0, lse = scale q.k_0. Zero query: O = mean of V, lse = log n_k."""
    q, k, v = rand_head(40, 8, 5)
    O, lse = orc.decode_split_head(q[:2], k[:1], v[:1], 0.5, 3)
    assert np.allclose(O, np.repeat(v[:1], 2, axis=0), atol=1e-15)
    assert np.allclose(lse, 0.5 * (q[:2] @ k[0]), atol=1e-14)
    O, lse = orc.decode_split_head(np.zeros((1, 8)), k, v, 0.5, 6)
    assert np.allclose(O[0], v.mean(axis=0), atol=1e-14) and np.isclose(lse[0], np.log(40))


# ------------------------------------------------------------------ invariants

def rand_head(n, d, seed, dv=None):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, d)), rng.standard_normal((n, d)),
            rng.standard_normal((n, dv or d)))


@pytest.mark.parametrize("causal", [False, True])
def test_convex_combination(causal):
    q, k, v = rand_head(64, 16, 4)
    O, _ = orc.forward_head(q * 3, k, v, 0.25, causal=causal)
    for i in range(64):
        allowed = v[: i + 1] if causal else v
        assert np.all(O[i] <= allowed.max(axis=0) + 1e-12)
        assert np.all(O[i] >= allowed.min(axis=0) - 1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_scores_give_mean_of_values(causal):
    n = 50
    _, k, v = rand_head(n, 8, 5)
    O, lse = orc.forward_head(np.zeros((n, 8)), k, v, 0.125, causal=causal)
    if causal:
        want = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
        want_lse = np.log(np.arange(1, n + 1))
    else:
        want = np.broadcast_to(v.mean(axis=0), v.shape)
        want_lse = np.full(n, np.log(n))
    assert np.allclose(O, want, atol=1e-14)
    assert np.allclose(lse, want_lse, atol=1e-14)


def test_single_key_and_first_causal_row():
    q, k, v = rand_head(1, 8, 6)
    O, lse = orc.forward_head(q, k, v, 0.7)
    assert np.allclose(O, v, atol=0)
    assert np.isclose(lse[0], 0.7 * float(q[0] @ k[0]), atol=1e-15)
    q, k, v = rand_head(10, 8, 7)
    O, lse = orc.forward_head(q, k, v, 0.7, causal=True)
    assert np.array_equal(O[0], v[0])
    assert np.isclose(lse[0], 0.7 * float(q[0] @ k[0]), atol=1e-15)


def test_joint_key_value_permutation_invariance():
    q, k, v = rand_head(40, 12, 8)
    perm = np.random.default_rng(9).permutation(40)
    O, lse = orc.forward_head(q, k, v, 0.3)
    O2, lse2 = orc.forward_head(q, k[perm], v[perm], 0.3)
    assert np.allclose(O, O2, atol=1e-14)
    assert np.allclose(lse, lse2, atol=1e-14)


def test_all_ones_block_mask_equals_dense_and_diagonal_mask_is_blockwise():
    q, k, v = rand_head(32, 8, 10)
    O, lse = orc.forward_head(q, k, v, 0.5)
    Ob, lseb = orc.forward_head(q, k, v, 0.5, block_mask=np.ones((4, 4), np.uint8), tile=8)
    assert np.array_equal(O, Ob) and np.array_equal(lse, lseb)
    Od, lsed = orc.forward_head(q, k, v, 0.5, block_mask=np.eye(4, dtype=np.uint8), tile=8)
    for t in range(4):
        sl = slice(8 * t, 8 * t + 8)
        Ot, lt = orc.forward_head(q[sl], k[sl], v[sl], 0.5)
        assert np.allclose(Od[sl], Ot, atol=1e-14) and np.allclose(lsed[sl], lt, atol=1e-14)


def test_empty_rows_convention():
    q, k, v = rand_head(16, 4, 11)
    bm = np.array([[0, 1], [0, 1]], dtype=np.uint8)  # no query attends to keys 0..7
    O, lse = orc.forward_head(q, k, v, 1.0, block_mask=np.array([[0, 0], [0, 1]], np.uint8), tile=8)
    assert np.all(O[:8] == 0) and np.all(np.isneginf(lse[:8]))
    O2, _ = orc.forward_online_head(q, k, v, 1.0, block=3,
                                    block_mask=np.array([[0, 0], [0, 1]], np.uint8), tile=8)
    assert np.allclose(O, O2, atol=1e-14)
    O3, _ = orc.forward_head(q, k, v, 1.0, block_mask=bm, tile=8)
    O4, _ = orc.forward_head(q, k[8:], v[8:], 1.0)
    assert np.allclose(O3, O4, atol=1e-14)


# ------------------------------------------------------------------ online recurrence == definition

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block", [1, 2, 7, 128, 300])
def test_online_equals_definition_any_block(block, causal):
    q, k, v = rand_head(300, 32, 12)
    O, lse = orc.forward_head(q * 2, k, v, 1 / np.sqrt(32), causal=causal)
    O2, lse2 = orc.forward_online_head(q * 2, k, v, 1 / np.sqrt(32), block=block, causal=causal)
    assert np.max(np.abs(O - O2)) <= 1e-12
    assert np.max(np.abs(lse - lse2)) <= 1e-12


def test_online_with_block_mask_equals_definition():
    q, k, v = rand_head(64, 8, 13)
    bm = (np.random.default_rng(14).random((8, 8)) < 0.3).astype(np.uint8)
    np.fill_diagonal(bm, 1)
    O, lse = orc.forward_head(q, k, v, 0.4, block_mask=bm, tile=8)
    O2, lse2 = orc.forward_online_head(q, k, v, 0.4, block=5, block_mask=bm, tile=8)
    assert np.max(np.abs(O - O2)) <= 1e-12 and np.max(np.abs(lse - lse2)) <= 1e-12


@pytest.mark.parametrize("block", [1, 3, 16, 64])
def test_fa1_form_equals_fa2_form(block):
    q, k, v = rand_head(64, 16, 15)
    O, lse = orc.forward_online_head(q, k, v, 0.25, block=block)
    O1, lse1 = orc.forward_fa1_head(q, k, v, 0.25, block=block)
    assert np.max(np.abs(O - O1)) <= 1e-12 and np.max(np.abs(lse - lse1)) <= 1e-12


def test_batched_forward_matches_per_head():
    rng = np.random.default_rng(16)
    q, k, v = (rng.standard_normal((2, 3, 20, 8)) for _ in range(3))
    O, lse = orc.forward(q, k, v, 0.35, causal=True)
    for b in range(2):
        for h in range(3):
            Oh, lh = orc.forward_head(q[b, h], k[b, h], v[b, h], 0.35, causal=True)
            assert np.array_equal(O[b, h], Oh) and np.array_equal(lse[b, h], lh)
    # sampled rows use the same definition
    Or, lr = orc.forward_head(q[1, 2], k[1, 2], v[1, 2], 0.35, causal=True, rows=[0, 7, 19])
    assert np.array_equal(Or, O[1, 2, [0, 7, 19]]) and np.array_equal(lr, lse[1, 2, [0, 7, 19]])


# ------------------------------------------------------------------ backward

def loss(q, k, v, do, scale, causal, bm=None, tile=4):
    O, _ = orc.forward_head(q, k, v, scale, causal=causal, block_mask=bm, tile=tile)
    return float((O * do).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    n, d = 12, 6
    rng = np.random.default_rng(17)
    q, k, v, do = (rng.standard_normal((n, d)) for _ in range(4))
    scale = 0.6
    dq, dk, dv = orc.backward_head(q, k, v, do, scale, causal=causal)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"], do, scale, causal)
                        - loss(args_m["q"], args_m["k"], args_m["v"], do, scale, causal)) / (2 * h)
        assert np.max(np.abs(num - g)) < 1e-7 * max(1.0, np.max(np.abs(g))), name


@pytest.mark.parametrize("n,causal", [(12, False), (10, True)])
def test_backward_block_mask_matches_finite_differences(n, causal):
    """Tile mask alone, and combined with the causal mask on a ragged size (last tile 2 rows)."""
    d, tile = 4, 4
    rng = np.random.default_rng(18)
    q, k, v, do = (rng.standard_normal((n, d)) for _ in range(4))
    bm = np.array([[1, 0, 1], [0, 1, 0], [1, 1, 1]], np.uint8)
    dq, dk, dv = orc.backward_head(q, k, v, do, 0.5, causal=causal, block_mask=bm, tile=tile)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            a_p = {"q": q, "k": k, "v": v, name: xp}
            a_m = {"q": q, "k": k, "v": v, name: xm}
            num[idx] = (loss(a_p["q"], a_p["k"], a_p["v"], do, 0.5, causal, bm, tile)
                        - loss(a_m["q"], a_m["k"], a_m["v"], do, 0.5, causal, bm, tile)) / (2 * h)
        assert np.max(np.abs(num - g)) < 1e-7 * max(1.0, np.max(np.abs(g))), name


@pytest.mark.parametrize("causal", [False, True])
def test_backward_invariants(causal):
    q, k, v = rand_head(48, 16, 19)
    do = np.random.default_rng(20).standard_normal((48, 16))
    dq, dk, dv = orc.backward_head(q, k, v, do, 0.25, causal=causal)
    # rows of dS sum to zero  =>  sum_j dK_j = 0;  rows of P sum to one  =>  sum_j dV_j = sum_i dO_i
    assert np.allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    assert np.allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-12)
    # a constant shift of all keys changes no score difference within a row, hence no output:
    # the derivative of L along k -> k + t*1 is zero for every direction c
    c = np.random.default_rng(21).standard_normal(16)
    assert abs(float((dk @ c).sum())) < 1e-12


@pytest.mark.parametrize("n,causal,masked", [(11, False, False), (10, True, True)])
def test_backward_sampled_matches_finite_differences(n, causal, masked):
    """The row-blocked backward of sampled query rows and key columns (blocks of 3 rows, so that
    several blocks add into each dK, dV column), against central differences of L = sum(O * dO),
    ragged and with the tile mask and causal mask combined."""
    d, tile = 4, 4
    rng = np.random.default_rng(23)
    q, k, v, do = (rng.standard_normal((n, d)) for _ in range(4))
    bm = np.array([[1, 0, 1], [1, 1, 0], [1, 1, 1]], np.uint8) if masked else None
    rows, cols = np.array([0, 4, n - 1]), np.array([1, 5, n - 2])
    dq, dk, dv = orc.backward_head_sampled(q, k, v, do, 0.5, rows, cols, causal=causal,
                                           block_mask=bm, tile=tile, row_block=3)
    h = 1e-6
    for name, x, g, idx_rows in (("q", q, dq, rows), ("k", k, dk, cols), ("v", v, dv, cols)):
        num = np.zeros_like(g)
        for a_i, r in enumerate(idx_rows):
            for c in range(d):
                xp, xm = x.copy(), x.copy()
                xp[r, c] += h
                xm[r, c] -= h
                a_p = {"q": q, "k": k, "v": v, name: xp}
                a_m = {"q": q, "k": k, "v": v, name: xm}
                num[a_i, c] = (loss(a_p["q"], a_p["k"], a_p["v"], do, 0.5, causal, bm, tile)
                               - loss(a_m["q"], a_m["k"], a_m["v"], do, 0.5, causal, bm, tile)) / (2 * h)
        assert np.max(np.abs(num - g)) < 1e-7 * max(1.0, np.max(np.abs(g))), name


def test_backward_sampled_invariants():
    """Every row and column sampled: rows of dS sum to zero and rows of P to one, so the key
    columns of dK sum to zero and those of dV to the column sums of dO."""
    q, k, v = rand_head(40, 8, 24)
    do = np.random.default_rng(25).standard_normal((40, 8))
    allr = np.arange(40)
    dq, dk, dv = orc.backward_head_sampled(q, k, v, do, 0.3, allr, allr, causal=True, row_block=7)
    assert np.allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    assert np.allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-12)


def test_backward_batched_matches_per_head():
    rng = np.random.default_rng(22)
    q, k, v, do = (rng.standard_normal((1, 2, 10, 4)) for _ in range(4))
    dq, dk, dv = orc.backward(q, k, v, do, 0.5, causal=True)
    for h in range(2):
        a, b, c = orc.backward_head(q[0, h], k[0, h], v[0, h], do[0, h], 0.5, causal=True)
        assert np.array_equal(dq[0, h], a) and np.array_equal(dk[0, h], b) and np.array_equal(dv[0, h], c)


# ------------------------------------------------------------------ planted mistakes are caught

def test_pins_catch_a_dropped_rescale(golden, monkeypatch):
    """A recurrence without the alpha correction would fail the figure-2 pin."""
    g = golden["figure2_chunked_update"]
    q, k = scores_as_attention(g["scores"])
    v = np.asarray(g["values"], dtype=np.float64)
    real_exp = np.exp
    calls = {"n": 0}

    def exp_without_correction(x):  # plant the mistake in the oracle: alpha forced to 1
        calls["n"] += 1
        y = real_exp(x)
        if np.ndim(x) == 1 and calls["n"] % 2 == 1:
            return np.ones_like(y)
        return y

    monkeypatch.setattr(orc.np, "exp", exp_without_correction)
    O, _ = orc.forward_online_head(q, k, v, 1.0, block=2)
    monkeypatch.setattr(orc.np, "exp", real_exp)
    assert not np.allclose(O[0], g["output"], atol=PRINTED_TOL)
