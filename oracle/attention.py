"""Plain fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg and its
reference arm) may import this module. The library and its Python binding never call it; the
oracle shares no code with the CUDA path (the two meet only in the seeded input generator, which
holds no attention arithmetic).

Sources (cited below by the short names in brackets):

* [TLDR]   tech-tldr.com, "FlashAttention：メモリ効率的なアテンション計算" -- sections
           "オンライン softmax" (running max / sum / output with correction factor alpha) and
           "タイル化" (outer loop over Q blocks, inner loop over K/V blocks, one division at the end).
* [XYZ]    xyznot.com, "FlashAttention: IOを意識した高速かつメモリ効率の高い厳密なアテンション"
           (summary of arXiv 2205.14135) -- "手法": statistics merge of m and l, steps 1-4 of the
           per-block update (FA1 form); "拡張: Block-Sparse FlashAttention" (tile mask M).
* [REAPER] mkdocs.reaper.mx, "3 · FlashAttention" -- 3.1 (S = QK^T/sqrt(d_h), P = softmax(S),
           O = PV), 3.3 "Le softmax en ligne", 3.4 (backward recomputes P from (m, l)), Q&A on the
           causal mask (query block i only needs key blocks j <= i).
* [LLMSE]  llm-systems-engineering.pages.dev, "출력을 누적해 메모리 이동을 줄이는 FlashAttention" --
           figure 1 (deferred normalisation), figure 2 (chunked update of l and a), figure 3
           (2 queries x 4 keys tile walk-through); FlashAttention-2 order of operations.
* [Q67]    quant67.com, "FlashAttention：在线 softmax 与 IO-aware 注意力" -- section 二 (block
           recurrence), section 五 (backward keeps O, m, l and recomputes P).

Plain definition implemented here (every function below reaches exactly this result up to
floating-point rounding order):

    S = scale * Q K^T,  S_ij = -inf where masked (causal: key j > query i; block-sparse:
    M[i // 128][j // 128] == 0),  m_i = max_j S_ij,  P_ij = exp(S_ij - m_i) / sum_j exp(S_ij - m_i),
    O = P V,  lse_i = m_i + ln sum_j exp(S_ij - m_i).

The pages do not spell out the gradients; the backward is standard softmax calculus applied to the
definition above (P recomputed from the inputs, as the pages prescribe):

    dV = P^T dO,  dP = dO V^T,  D_i = sum_k dO_ik O_ik,  dS = P * (dP - D),
    dQ = scale * dS K,  dK = scale * dS^T Q.

Readings where the pages leave a point open: the saved statistic is the natural-log logsumexp of
the *scaled* scores (one number per row instead of the pages' pair (m, l)); a row whose keys are
all masked has O = 0 and lse = -inf; the block mask is shared by all (batch, head) pairs.

Every function has a pin in tests/test_oracle_pins.py (worked examples of [LLMSE], scipy's
softmax/logsumexp as special cases, invariants, finite differences for the backward).
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


# ----------------------------------------------------------------------------------------------
# masks
# ----------------------------------------------------------------------------------------------

def allowed_keys(rows: np.ndarray, n_keys: int, causal: bool = False,
                 block_mask: np.ndarray | None = None, tile: int = 128) -> np.ndarray:
    """Boolean [len(rows), n_keys]: True where query ``rows[r]`` may attend to key j.

    Causal ([REAPER] Q&A on the causal mask): key j is allowed for query i iff j <= i.
    Block-sparse ([XYZ] "Block-Sparse FlashAttention"): only tiles with M[i//tile][j//tile] = 1.
    """
    rows = np.asarray(rows)
    keys = np.arange(n_keys)
    ok = np.ones((rows.size, n_keys), dtype=bool)
    if causal:
        ok &= keys[None, :] <= rows[:, None]
    if block_mask is not None:
        bm = np.asarray(block_mask).astype(bool)
        ok &= bm[rows // tile][:, keys // tile]
    return ok


# ----------------------------------------------------------------------------------------------
# the plain definition ([REAPER] 3.1, [TLDR] first formula, [Q67] section 一)
# ----------------------------------------------------------------------------------------------

def softmax_rows(S: np.ndarray, ok: np.ndarray):
    """Max-subtracted softmax of each row of S over the allowed entries.

    Returns (P, lse). Rows with no allowed entry get P = 0 and lse = -inf.
    """
    S = np.where(ok, S, NEG_INF)
    m = S.max(axis=1)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    E = np.exp(S - m_safe[:, None])  # exp(-inf) = 0 on masked entries
    ell = E.sum(axis=1)
    ell_safe = np.where(empty, 1.0, ell)
    P = E / ell_safe[:, None]
    lse = np.where(empty, NEG_INF, m_safe + np.log(ell_safe))
    return P, lse


def forward_head(q, k, v, scale, causal=False, block_mask=None, tile=128, rows=None,
                 row_block=1024):
    """O and lse of one head by the plain definition (materialises S and P).

    ``rows`` restricts the computation to some query rows (rows are independent, so this is the
    same computation). Large heads are processed ``row_block`` query rows at a time for the same
    reason.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_keys = k.shape[0]
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    O = np.empty((rows.size, v.shape[1]))
    lse = np.empty(rows.size)
    for r0 in range(0, rows.size, row_block):
        rr = rows[r0:r0 + row_block]
        S = scale * (q[rr] @ k.T)
        P, l = softmax_rows(S, allowed_keys(rr, n_keys, causal, block_mask, tile))
        O[r0:r0 + rr.size] = P @ v
        lse[r0:r0 + rr.size] = l
    return O, lse


def forward(q, k, v, scale, causal=False, block_mask=None, tile=128):
    """Batched plain-definition forward over [B, H, N, d] arrays; returns (O, lse[B, H, N])."""
    B, H, N, _ = q.shape
    O = np.empty(q.shape[:3] + (v.shape[3],))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            O[b, h], lse[b, h] = forward_head(q[b, h], k[b, h], v[b, h], scale, causal,
                                              block_mask, tile)
    return O, lse


# ----------------------------------------------------------------------------------------------
# the online recurrence, for self-checks of the definition
# ----------------------------------------------------------------------------------------------

def forward_online_head(q, k, v, scale, block, causal=False, block_mask=None, tile=128,
                        trace=None):
    """Chunked online softmax with deferred normalisation (FlashAttention-2 order).

    Follows [TLDR] "オンライン softmax" / [LLMSE] figure 2 / [Q67] section 二: for each block of
    ``block`` keys, m_new = max(m, rowmax S_blk); alpha = exp(m - m_new); l = l*alpha + rowsum
    exp(S_blk - m_new); a = a*alpha + exp(S_blk - m_new) V_blk; m = m_new. At the end O = a / l.
    If ``trace`` is a list, the state (m, l, a) after each block is appended to it.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_q, n_k = q.shape[0], k.shape[0]
    rows = np.arange(n_q)
    m = np.full(n_q, NEG_INF)
    ell = np.zeros(n_q)
    a = np.zeros((n_q, v.shape[1]))
    for j0 in range(0, n_k, block):
        j1 = min(n_k, j0 + block)
        S = scale * (q @ k[j0:j1].T)
        ok = allowed_keys(rows, n_k, causal, block_mask, tile)[:, j0:j1]
        S = np.where(ok, S, NEG_INF)
        m_new = np.maximum(m, S.max(axis=1))
        live = np.isfinite(m_new)
        m_ref = np.where(live, m_new, 0.0)
        # exp(-inf - m_new) = 0 when nothing was accumulated yet; 1 while the row is still empty
        alpha = np.where(live, np.exp(m - m_ref), 1.0)
        E = np.exp(S - m_ref[:, None])
        ell = ell * alpha + E.sum(axis=1)
        a = a * alpha[:, None] + E @ v[j0:j1]
        m = m_new
        if trace is not None:
            trace.append((m.copy(), ell.copy(), a.copy()))
    empty = ell == 0.0
    O = a / np.where(empty, 1.0, ell)[:, None]
    lse = np.full(n_q, NEG_INF)
    lse[~empty] = m[~empty] + np.log(ell[~empty])
    return O, lse


def forward_fa1_head(q, k, v, scale, block):
    """The FlashAttention-1 per-block update ([XYZ] "手法" steps 1-4), dense, for cross-checks.

    Per key block j: m~ = rowmax S_j, P~ = exp(S_j - m~), l~ = rowsum P~; m_new = max(m, m~);
    l_new = e^(m - m_new) l + e^(m~ - m_new) l~;
    O <- diag(l_new)^-1 (diag(l) e^(m - m_new) O + e^(m~ - m_new) P~ V_j).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_q = q.shape[0]
    m = np.full(n_q, NEG_INF)
    ell = np.zeros(n_q)
    O = np.zeros((n_q, v.shape[1]))
    for j0 in range(0, k.shape[0], block):
        S = scale * (q @ k[j0:j0 + block].T)
        m_t = S.max(axis=1)
        P_t = np.exp(S - m_t[:, None])
        l_t = P_t.sum(axis=1)
        m_new = np.maximum(m, m_t)
        c_old = np.where(np.isfinite(m), np.exp(m - m_new), 0.0)
        c_new = np.exp(m_t - m_new)
        l_new = c_old * ell + c_new * l_t
        O = ((ell * c_old)[:, None] * O + c_new[:, None] * (P_t @ v[j0:j0 + block])) / l_new[:, None]
        m, ell = m_new, l_new
    return O, m + np.log(ell)


def decode_split_head(q, k, v, scale, n_splits):
    """Flash-Decoding ([REAPER] 3.6 "L'attention en décodage" and the Flash-Decoding row of 3.7):
    the keys are cut into ``n_splits`` contiguous chunks of ceil(n_k / n_splits) keys, each chunk
    gives (O_c, lse_c) by the plain definition, and the chunks are combined with the softmax
    statistics merge ([XYZ] "手法", merge of (m, l); [REAPER] 3.3):
    lse = log sum_c exp(lse_c),  O = sum_c exp(lse_c - lse) O_c.
    A chunk past the end of the keys is empty (lse_c = -inf) and gets weight 0.
    """
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_q, n_k = np.asarray(q).shape[0], k.shape[0]
    per = -(-n_k // n_splits)
    parts = []
    for c in range(n_splits):
        j0, j1 = c * per, min(n_k, (c + 1) * per)
        if j0 >= j1:
            parts.append((np.zeros((n_q, v.shape[1])), np.full(n_q, NEG_INF)))
        else:
            parts.append(forward_head(q, k[j0:j1], v[j0:j1], scale))
    L = np.stack([p[1] for p in parts])  # [n_splits, n_q]
    top = L.max(axis=0)
    W = np.exp(L - top[None, :])
    den = W.sum(axis=0)
    O = sum(W[c][:, None] * parts[c][0] for c in range(n_splits)) / den[:, None]
    return O, top + np.log(den)


# ----------------------------------------------------------------------------------------------
# backward ([REAPER] 3.4, [Q67] section 五: recompute P from the inputs; gradients by calculus)
# ----------------------------------------------------------------------------------------------

def backward_head(q, k, v, do, scale, causal=False, block_mask=None, tile=128):
    """dQ, dK, dV of L = sum(O * dO) for one head, by the plain definition (materialises P)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    rows = np.arange(q.shape[0])
    S = scale * (q @ k.T)
    P, _ = softmax_rows(S, allowed_keys(rows, k.shape[0], causal, block_mask, tile))
    O = P @ v
    dV = P.T @ do
    dP = do @ v.T
    D = (do * O).sum(axis=1)
    dS = P * (dP - D[:, None])
    dQ = scale * (dS @ k)
    dK = scale * (dS.T @ q)
    return dQ, dK, dV


def backward_head_sampled(q, k, v, do, scale, rows, cols, causal=False, block_mask=None, tile=128,
                          row_block=1024):
    """dQ at query ``rows`` and dK, dV at key ``cols`` of one head, by the same definition as
    ``backward_head`` without materialising the whole N x N P: the query rows are walked
    ``row_block`` at a time, each block's P (and O, D) formed in full, and only the sampled
    columns of dS and P kept. dQ rows are independent of each other; a key column of dK or dV
    sums over every query row, which every block contributes to.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    rows = np.asarray(rows)
    cols = np.asarray(cols)
    n = q.shape[0]
    dq = np.zeros((rows.size, q.shape[1]))
    dk = np.zeros((cols.size, k.shape[1]))
    dv = np.zeros((cols.size, v.shape[1]))
    for r0 in range(0, n, row_block):
        rr = np.arange(r0, min(n, r0 + row_block))
        S = scale * (q[rr] @ k.T)
        P, _ = softmax_rows(S, allowed_keys(rr, k.shape[0], causal, block_mask, tile))
        O = P @ v
        D = (do[rr] * O).sum(axis=1)
        Pc = P[:, cols]
        dSc = Pc * (do[rr] @ v[cols].T - D[:, None])
        dv += Pc.T @ do[rr]
        dk += scale * (dSc.T @ q[rr])
        sel = np.nonzero((rows >= r0) & (rows < r0 + rr.size))[0]
        if sel.size:
            lr = rows[sel] - r0
            dS = P[lr] * (do[rows[sel]] @ v.T - D[lr][:, None])
            dq[sel] = scale * (dS @ k)
    return dq, dk, dv


def backward(q, k, v, do, scale, causal=False, block_mask=None, tile=128):
    """Batched backward over [B, H, N, d] arrays; returns (dQ, dK, dV)."""
    dq = np.empty(q.shape)
    dk = np.empty(k.shape)
    dv = np.empty(v.shape)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            dq[b, h], dk[b, h], dv[b, h] = backward_head(q[b, h], k[b, h], v[b, h], do[b, h],
                                                         scale, causal, block_mask, tile)
    return dq, dk, dv
