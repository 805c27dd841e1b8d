"""Pins of the oracle's Lightning Indexer scores and Top-K: a hand-computed 2-head /
8-position example (with ReLU cut-offs, a zero weight, negative weights, exact ties and
the causal cut), a second route through torch.einsum, brute-force stable sorting and the
selection invariants."""

import numpy as np
import pytest
import torch

from oracle.quant import mxfp8_quantize, mxfp8_dequantize
from oracle.indexer import (indexer_scores_row, indexer_magnitude_row, topk_row, selectable_count,
                            indexer_topk_rows)
from oracle.pipeline import decode_rows

# Hand example (tests/golden/indexer_hand_2h8p.json): only the first four of the 128
# dims are non-zero and every value is a small integer, so MXFP8 quantisation is exact and
# the scores follow by hand.
import json
import os

_G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "indexer_hand_2h8p.json")))
Q = np.zeros((2, 128))
Q[:, :4] = _G["q_dims0_3"]
K8 = np.zeros((8, 128))
K8[:, :4] = _G["k_dims0_3"]
CASES = _G["cases"]


def _deq(x):
    c, s = mxfp8_quantize(x)
    return mxfp8_dequantize(c, s)


def test_hand_example_quantisation_is_exact():
    assert np.array_equal(_deq(Q), Q) and np.array_equal(_deq(K8), K8)


def test_hand_dots():
    assert (_deq(K8) @ _deq(Q).T).tolist() == _G["dots"]


@pytest.mark.parametrize("case", CASES)
def test_hand_scores(case):
    s = indexer_scores_row(_deq(Q), np.array(case["w"]), _deq(K8))
    assert s.tolist() == case["scores"]


@pytest.mark.parametrize("case", CASES)
def test_hand_magnitude(case):
    # the denominator of every score tolerance and of the Top-K tie band: hand values that
    # a dropped abs on w, an abs taken after the head sum, or a ReLU applied to it would miss
    m = indexer_magnitude_row(_deq(Q), np.array(case["w"]), _deq(K8))
    assert m.tolist() == case["magnitude"]


def test_magnitude_bounds_score():
    # |score| <= magnitude always, with equality when every weight and dot is >= 0
    rng = np.random.default_rng(5)
    q, k, w = rng.standard_normal((4, 128)), rng.standard_normal((50, 128)), rng.standard_normal(4)
    s, m = indexer_scores_row(q, w, k), indexer_magnitude_row(q, w, k)
    assert np.all(np.abs(s) <= m * (1 + 1e-12))
    qp, kp, wp = np.abs(q), np.abs(k), np.abs(w)
    assert np.allclose(indexer_scores_row(qp, wp, kp), indexer_magnitude_row(qp, wp, kp), rtol=1e-12)


@pytest.mark.parametrize("case", CASES)
def test_hand_topk(case):
    s = indexer_scores_row(_deq(Q), np.array(case["w"]), _deq(K8))
    for k, want in case["topk"].items():
        idx, _ = topk_row(s, int(k))
        assert idx.tolist() == want


def test_hand_causal_cut():
    # query at position 5 may select p0..p5 only
    n = selectable_count(5, 8)
    assert n == 6
    idx, _, _ = indexer_topk_rows(_deq(Q)[None], np.array([CASES[0]["w"]]), [_deq(K8)], [n], 3)
    assert idx[0].tolist() == CASES[0]["causal_pos5_top3"]
    assert selectable_count(7, 8) == 8 and selectable_count(100, 8) == 8


def test_scores_vs_einsum_route():
    rng = np.random.default_rng(0)
    q = _deq(rng.standard_normal((64, 128)))
    k = _deq(rng.standard_normal((300, 128)))
    w = rng.standard_normal(64) / 8
    ref = torch.einsum("hd,pd->ph", torch.from_numpy(q), torch.from_numpy(k)).clamp_min(0) @ torch.from_numpy(w)
    assert np.allclose(indexer_scores_row(q, w, k), ref.numpy(), rtol=1e-13, atol=1e-13)


def test_topk_vs_bruteforce_sort_with_many_ties():
    rng = np.random.default_rng(1)
    for trial in range(200):
        n = int(rng.integers(1, 60))
        s = rng.integers(-4, 5, n).astype(np.float64)    # many exact ties
        k = int(rng.integers(1, 70))
        want = sorted(range(n), key=lambda p: (-s[p], p))[:k]
        want += [-1] * (k - len(want))
        idx, vals = topk_row(s, k)
        assert idx.tolist() == want
        sel = idx[idx >= 0]
        # invariants: every selected score >= every unselected one
        rest = np.setdiff1d(np.arange(n), sel)
        if rest.size and sel.size:
            assert s[sel].min() >= s[rest].max()
        assert len(set(sel.tolist())) == sel.size == min(k, n)


def test_pipeline_rows_shapes_and_causality():
    rng = np.random.default_rng(2)
    L = 200
    k = rng.standard_normal((L, 128))
    kv = rng.standard_normal((L, 576))
    qi = rng.standard_normal((2, 8, 128))
    w = rng.standard_normal((2, 8))
    qs = rng.standard_normal((2, 4, 576))
    out = decode_rows([0, 1], qi, w, [k, k], qs, [kv, kv], [150, 199], [L, L], 64, 0.1)
    assert all(i.max() <= p for i, p in zip(out["idx"], [150, 199]))
    assert out["o"][0].shape == (4, 512)
