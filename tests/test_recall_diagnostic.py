"""Synthetic Top-K recall of the MXFP8 indexer (a diagnostic, not a parity gate).

"Kimi K3.1 Pro Inference Acceleration: Day0 Optimization on Heterogeneous AI Hardware",
section "Full MXFP8 Quantization with Per-Group Dynamic Scaling for LI", reports that the
MXFP8 indexer (one scale per 32 elements) loses less than 0.1% Top-K recall against its
BF16 baseline on a long-sequence benchmark with trained weights.  Neither the benchmark
nor the weights exist here, so this measures the synthetic analogue on the benchmark
workloads' own inputs: the Top-K of the float64 oracle over MXFP8-quantised queries and
keys against the Top-K of the same oracle over the unquantised bf16 queries and keys.

Random N(0, 1) inputs make the scores of the selected band nearly equal, so quantisation
reorders many of them; the figures printed here are therefore far below the pages' trained
model figure and only a floor is asserted.  On the long-context workload with planted
keys (1% of the keys at cosine 0.5 to the first row's weighted query) the planted keys
stand out of the Top-K band of that row, and the recall there must be higher.
"""

import numpy as np
import pytest

import oracle
from dsa_sparse_attention_topk_gb300 import workloads as W


def _recall(wl, r, n_ctx=None):
    b = int(wl.q_seq[r])
    q = wl.q_index().double().numpy()[r]
    w = wl.weights().double().numpy()[r]
    n = oracle.indexer.selectable_count(wl.q_pos[r], wl.seq_lens[b])
    if n_ctx is not None:
        n = min(n, n_ctx)
    k = wl.k_seq(b).double().numpy()[:n]
    exact, _ = oracle.topk_row(oracle.indexer_scores_row(q, w, k), wl.topk)
    qh = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(q))
    kh = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(k))
    quant, _ = oracle.topk_row(oracle.indexer_scores_row(qh, w, kh), wl.topk)
    a, b_ = set(exact[exact >= 0].tolist()), set(quant[quant >= 0].tolist())
    return len(a & b_) / max(1, len(a)), a


@pytest.mark.parametrize("name", ["decode_b32_ctx32k", "mixed_b128"])
def test_mxfp8_topk_recall_on_random_inputs(name):
    wl = W.make(name)
    recalls = [_recall(wl, r)[0] for r in (0, wl.n_q // 2)]
    print(f"{name}: MXFP8 vs unquantised Top-{wl.topk} recall {', '.join(f'{x:.3f}' for x in recalls)}")
    assert min(recalls) > 0.7


def test_mxfp8_keeps_the_planted_keys():
    wl = W.make("long_mtp_b4_ctx128k")
    rec, exact = _recall(wl, 0, n_ctx=32768)   # the first 32K positions of row 0's sequence
    print(f"long_mtp_b4_ctx128k row 0 (first 32K positions): recall {rec:.3f}")
    assert rec > 0.95
