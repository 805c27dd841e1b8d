"""The whole DSA decode path for chosen query rows, on logical (unpaged) tensors.
Test infrastructure only.

Order of the steps follows "Kimi K3.1 Pro Inference Acceleration: Day0 Optimization on
Heterogeneous AI Hardware" (sections "Lightning Indexer Three-Stream Coordination",
"Full MXFP8 Quantization ...", "FP8 KVCache ...") and "Deep Dive into Sparse Attention
..." section 1: quantise the indexer query (MXFP8) and the caches (MXFP8 k, FP8 latent
kv), score every selectable position, keep the Top-K, then run Sparse Flash Attention
over the selected latent rows.
"""

import numpy as np

from .quant import mxfp8_quantize, mxfp8_dequantize, fp8_tile_quantize, fp8_tile_dequantize
from .indexer import indexer_scores_row, topk_row, selectable_count
from .sfa import sparse_attention_row


def decode_rows(rows, q_idx, w, k_seq, q_sfa, kv_seq, q_pos, seq_len, topk, sm_scale,
                want_scores=False):
    """Run the path for a list of query rows.

    rows: iterable of row ids; q_idx[r] (H_I, 128) bf16 values; w[r] (H_I,);
    k_seq[r] (ctx_r, 128) bf16 values of the row's sequence; q_sfa[r] (H_S, 576);
    kv_seq[r] (ctx_r, 576); q_pos[r], seq_len[r] ints.  Arrays may be any float type
    holding the exact bf16 values; everything is computed in float64.

    Returns dict of per-row lists: idx (topk,), vals, o (H_S, 512), lse (H_S,), and the
    full score vector when want_scores.
    """
    out = {"idx": [], "vals": [], "o": [], "lse": [], "scores": []}
    for r in rows:
        n = selectable_count(q_pos[r], seq_len[r])
        qc, qs = mxfp8_quantize(np.asarray(q_idx[r], np.float64))
        q_hat = mxfp8_dequantize(qc, qs)
        kc, ks = mxfp8_quantize(np.asarray(k_seq[r][:n], np.float64))
        k_hat = mxfp8_dequantize(kc, ks)
        s = indexer_scores_row(q_hat, np.asarray(w[r], np.float64), k_hat)
        idx, vals = topk_row(s, topk)
        sel = idx[idx >= 0]
        kv_rows = np.asarray(kv_seq[r], np.float64)
        # quantise only the selected latent rows: the tile rule is per token
        vc, vs = fp8_tile_quantize(kv_rows[sel]) if sel.size else (None, None)
        kv_hat = np.zeros((n, kv_rows.shape[1]))
        if sel.size:
            kv_hat[sel] = fp8_tile_dequantize(vc, vs)
        o, lse = sparse_attention_row(np.asarray(q_sfa[r], np.float64), kv_hat, idx, sm_scale)
        out["idx"].append(idx)
        out["vals"].append(vals)
        out["o"].append(o)
        out["lse"].append(lse)
        if want_scores:
            out["scores"].append(s)
    return out
