"""Pins of the oracle's Sparse Flash Attention: with every position selected it equals
dense attention (torch scaled_dot_product_attention in float64); a single selected entry
returns that entry's value row; a two-entry hand example; the lse normalises the weights;
order and -1 padding of the index list do not matter."""

import math

import numpy as np
import torch

from oracle.quant import fp8_tile_quantize, fp8_tile_dequantize
from oracle.sfa import sparse_attention_row
from oracle.pipeline import decode_rows
from oracle.quant import mxfp8_quantize, mxfp8_dequantize

SM = 1.0 / math.sqrt(192.0)


def _kvhat(n, seed):
    rng = np.random.default_rng(seed)
    c, s = fp8_tile_quantize(rng.standard_normal((n, 576)))
    return fp8_tile_dequantize(c, s)


def _dense(q, kvh, scale):
    qt = torch.from_numpy(q)[None, :, None, :]                    # (1, H, 1, 576)
    kt = torch.from_numpy(kvh)[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.from_numpy(kvh[:, :512])[None, None].expand(1, q.shape[0], -1, -1)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0, :, 0].numpy()


def test_all_selected_equals_dense_attention():
    rng = np.random.default_rng(0)
    kvh = _kvhat(77, 1)
    q = rng.standard_normal((16, 576))
    idx = np.concatenate([rng.permutation(77), -np.ones(13, int)])
    o, lse = sparse_attention_row(q, kvh, idx, SM)
    assert np.allclose(o, _dense(q, kvh, SM), rtol=1e-12, atol=1e-12)


def test_single_entry_returns_value_row():
    rng = np.random.default_rng(1)
    kvh = _kvhat(10, 2)
    q = rng.standard_normal((4, 576))
    o, lse = sparse_attention_row(q, kvh, np.array([-1, 6, -1]), SM)
    assert np.array_equal(o, np.broadcast_to(kvh[6, :512], o.shape))
    assert np.allclose(lse, SM * q @ kvh[6], rtol=1e-14)


def test_two_entry_hand_example():
    # logits 0 and log 3 -> weights 1/4, 3/4
    kv = np.zeros((2, 576))
    kv[0, :512] = 1.0
    kv[1, :512] = -1.0
    kv[1, 512] = 1.0
    q = np.zeros((1, 576))
    q[0, 512] = math.log(3.0)
    o, lse = sparse_attention_row(q, kv, np.array([0, 1]), 1.0)
    assert np.allclose(o[0], 0.25 * 1.0 + 0.75 * -1.0, rtol=0, atol=1e-15)
    assert math.isclose(lse[0], math.log(4.0), rel_tol=1e-15)


def test_lse_normalises_weights():
    rng = np.random.default_rng(3)
    kvh = _kvhat(50, 4)
    q = rng.standard_normal((8, 576))
    idx = rng.choice(50, 20, replace=False)
    o, lse = sparse_attention_row(q, kvh, idx, SM)
    p = np.exp(SM * q @ kvh[idx].T - lse[:, None])
    assert np.allclose(p.sum(1), 1.0, rtol=1e-13)
    assert np.allclose(p @ kvh[idx, :512], o, rtol=1e-12, atol=1e-13)


def test_order_and_padding_invariance():
    rng = np.random.default_rng(4)
    kvh = _kvhat(40, 5)
    q = rng.standard_normal((3, 576))
    idx = rng.choice(40, 15, replace=False)
    o1, l1 = sparse_attention_row(q, kvh, idx, SM)
    o2, l2 = sparse_attention_row(q, kvh, np.concatenate([[-1], idx[::-1], [-1, -1]]), SM)
    assert np.allclose(o1, o2, rtol=1e-13, atol=1e-14) and np.allclose(l1, l2, rtol=1e-13)


def test_empty_selection():
    o, lse = sparse_attention_row(np.ones((2, 576)), np.zeros((3, 576)), np.array([-1, -1]), SM)
    assert not o.any() and np.all(np.isneginf(lse))


def test_pipeline_topk_ge_n_is_dense_attention_over_prefix():
    # Top-K >= selectable count: the path reduces to dense causal attention over the
    # dequantised prefix
    rng = np.random.default_rng(6)
    L = 130
    k = rng.standard_normal((L, 128))
    kv = rng.standard_normal((L, 576))
    qi = rng.standard_normal((1, 8, 128))
    w = rng.standard_normal((1, 8))
    qs = rng.standard_normal((1, 16, 576))
    pos = 100
    out = decode_rows([0], qi, w, [k], qs, [kv], [pos], [L], 256, SM)
    c, s = fp8_tile_quantize(kv[:pos + 1])
    ref = _dense(qs[0], fp8_tile_dequantize(c, s), SM)
    assert np.allclose(out["o"][0], ref, rtol=1e-12, atol=1e-12)
    assert sorted(out["idx"][0][out["idx"][0] >= 0].tolist()) == list(range(pos + 1))
