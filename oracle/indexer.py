"""Lightning Indexer scores and Top-K selection, in float64.  Test infrastructure only.

Passages followed:

* "Deep Dive into Sparse Attention and Engineering Optimizations for Efficient Inference
  in Kimi K3.1 Pro", section 1: a lightweight indexer scores the relevance of every
  historical key for each query position and the Top-K most relevant positions are kept.
* "Kimi K3.1 Pro Inference Acceleration: Day0 Optimization on Heterogeneous AI
  Hardware", section "Lightning Indexer Three-Stream Coordination": the indexer performs
  relevance scoring, head-weight weighting and Top-K index selection.

The pages print no formula.  The reading adopted here is the plainest one that names both
steps, a per-head relevance score and a weighting of the heads, with no extra scale:

    score[t, p] = sum_h  w[t, h] * max(0, q_hat[t, h, :] . k_hat[p, :])

over the dequantised MXFP8 q_hat (per query row and indexer head) and k_hat (per cached
position), with no extra scale factor, for every position p <= pos(t) and p < seq_len.
Top-K keeps the K highest scores; equal scores are ordered by lower position first; when
fewer than K positions are selectable all of them are kept and the rest of the row is
padded with -1.
"""

import numpy as np


def selectable_count(q_pos, seq_len):
    """Number of positions a query row at position q_pos may select (causal rule)."""
    return int(max(0, min(int(q_pos) + 1, int(seq_len))))


def indexer_scores_row(q_hat, w, k_hat):
    """Scores of one query row against n cached positions.

    q_hat: (H, D) dequantised indexer query; w: (H,) head weights; k_hat: (n, D).
    Returns float64 (n,).
    """
    q_hat = np.asarray(q_hat, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    k_hat = np.asarray(k_hat, dtype=np.float64)
    dots = k_hat @ q_hat.T                 # (n, H): q_hat[h] . k_hat[p]
    return np.maximum(dots, 0.0) @ w       # sum_h w[h] * ReLU(dot)


def indexer_magnitude_row(q_hat, w, k_hat):
    """sum_h |w[h]| * |q_hat[h] . k_hat[p]|: the no-cancellation size of each score,
    used to judge relative error of near-zero scores."""
    dots = np.asarray(k_hat, np.float64) @ np.asarray(q_hat, np.float64).T
    return np.abs(dots) @ np.abs(np.asarray(w, np.float64))


def topk_row(scores, k):
    """Top-K of one row: K highest scores, ties -> lower position, -1 padding.

    scores: float64 (n,) over positions 0..n-1.  Returns (idx int32 (k,), vals float64
    (k,), with vals = -inf where idx = -1).  The order is by descending score, then
    ascending position.
    """
    s = np.asarray(scores, dtype=np.float64)
    n = s.shape[0]
    order = np.argsort(-s, kind="stable")  # stable: equal scores keep ascending position
    m = min(k, n)
    idx = np.full(k, -1, dtype=np.int32)
    vals = np.full(k, -np.inf, dtype=np.float64)
    idx[:m] = order[:m]
    vals[:m] = s[order[:m]]
    return idx, vals


def indexer_topk_rows(q_hat, w, k_hat_of_row, n_sel, k):
    """Scores + Top-K for several query rows.

    q_hat: (R, H, D); w: (R, H); k_hat_of_row: list of (n_r, D) dequantised caches (the
    row's sequence, already cut to its selectable prefix or longer); n_sel: (R,) number of
    selectable positions per row.  Returns (idx (R, k) int32, vals (R, k), scores list).
    """
    R = q_hat.shape[0]
    out_idx = np.full((R, k), -1, dtype=np.int32)
    out_val = np.full((R, k), -np.inf)
    all_scores = []
    for r in range(R):
        n = int(n_sel[r])
        s = indexer_scores_row(q_hat[r], w[r], k_hat_of_row[r][:n])
        out_idx[r], out_val[r] = topk_row(s, k)
        all_scores.append(s)
    return out_idx, out_val, all_scores
