"""Sparse Flash Attention over the selected entries of the MLA latent cache, in float64.
Test infrastructure only.

Passages followed:

* "Deep Dive into Sparse Attention and Engineering Optimizations for Efficient Inference
  in Kimi K3.1 Pro", section 1: SFA runs attention only over the key-value pairs of the
  positions the indexer selected, on top of Multi-Head Latent Attention.
* "Adapting and Optimizing Kimi K3.1 Pro for Long-Sequence Inference", section 2: the
  sparse attention core gathers the cache entries named by the indices of the previous
  step.
* "Kimi K3.1 Pro Inference Acceleration: Day0 Optimization on Heterogeneous AI
  Hardware", section "Preserving a Mixed-Precision Path": the query and the final
  attention weighting stay BF16; only the cache is FP8.

Reading adopted (absorbed MLA decode, the form the workloads' 576-wide latent with a
512-wide value implies): each selected position j
carries one dequantised latent row kv_hat[j] of width 576 that serves as the key, and
its first 512 entries serve as the value.  For query row t and head h over the valid
(non -1) selected entries J:

    l_j = sm_scale * q[t, h, :] . kv_hat[j, :]
    o[t, h, :] = sum_j exp(l_j - m) kv_hat[j, :512] / sum_j exp(l_j - m),  m = max_j l_j
    lse[t, h]  = m + log(sum_j exp(l_j - m))

An empty selection gives o = 0 and lse = -inf.
"""

import numpy as np

D_LATENT = 576
D_V = 512


def sparse_attention_row(q, kv_hat, idx, sm_scale):
    """One query row: q (H, 576) float64; kv_hat (n, 576) dequantised latent cache of the
    row's sequence; idx (K,) selected positions with -1 padding.  Returns (o (H, 512),
    lse (H,))."""
    q = np.asarray(q, dtype=np.float64)
    idx = np.asarray(idx)
    sel = idx[idx >= 0]
    H = q.shape[0]
    if sel.size == 0:
        return np.zeros((H, D_V)), np.full(H, -np.inf)
    kv = np.asarray(kv_hat, dtype=np.float64)[sel]          # (J, 576): the gather
    logits = float(sm_scale) * (q @ kv.T)                   # (H, J)
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    l = p.sum(axis=1, keepdims=True)
    o = (p @ kv[:, :D_V]) / l
    lse = (m + np.log(l))[:, 0]
    return o, lse
