"""Why Sparse Flash Attention keeps its query and its weights in BF16.

"Kimi K3.1 Pro Inference Acceleration: Day0 Optimization on Heterogeneous AI Hardware",
section "Preserving a Mixed-Precision Path", keeps the query and the final attention
weighting in BF16 and puts only the cache in FP8.  A block-scaled FP8 tensor-core Q K^T
would need the query in E4M3 as well (both MMA operands of one kind share the 8-bit
type).  These tests measure, on the decode workload's value distributions (N(0,1) bf16
query and latent rows, 2048 selected entries, 128 heads, FP8 latent cache with a scale
per 128-element tile), what that costs against the stated output gate (max-abs 2e-2,
mean-abs 2e-3 against the float64 result):

* an E4M3 query, scaled per (head, 128-wide tile) or per 32 elements (MXFP8), misses
  the gate on its own;
* the BF16 path the kernels take (latent values rounded once to bf16, bf16 weights,
  fp32 sums) stays an order of magnitude inside it.
Everything here is float64 numpy on the CPU; the roundings are modelled exactly.
"""

import numpy as np
import pytest
import torch

import oracle

SFA_MAX_ABS = 2e-2
SFA_MEAN_ABS = 2e-3
SM_SCALE = 1.0 / np.sqrt(192.0)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).double().numpy()


@pytest.fixture(scope="module")
def row():
    rng = np.random.default_rng(20261203)
    q = _bf16(rng.standard_normal((128, 576)))
    kv = _bf16(rng.standard_normal((2048, 576)))
    c, s = oracle.fp8_tile_quantize(kv)
    kvh = oracle.fp8_tile_dequantize(c, s)
    idx = np.arange(2048)
    o_ref, _ = oracle.sparse_attention_row(q, kvh, idx, SM_SCALE)
    return q, kvh, idx, o_ref


def _err(o, o_ref):
    d = np.abs(o - o_ref)
    return d.max(), d.mean()


@pytest.mark.parametrize("fmt", ["e4m3_tile128", "mxfp8"])
def test_fp8_query_misses_the_output_gate(row, fmt):
    q, kvh, idx, o_ref = row
    if fmt == "e4m3_tile128":
        c, s = oracle.fp8_tile_quantize(q)
        qh = oracle.fp8_tile_dequantize(c, s)
    else:
        c, s = oracle.mxfp8_quantize(q)
        qh = oracle.mxfp8_dequantize(c, s)
    o, _ = oracle.sparse_attention_row(qh, kvh, idx, SM_SCALE)
    mx, mean = _err(o, o_ref)
    assert mean > SFA_MEAN_ABS, f"mean-abs {mean:.3e}"


def test_bf16_path_is_well_inside_the_gate(row):
    q, kvh, idx, o_ref = row
    kvb = _bf16(kvh)
    lg = SM_SCALE * (q @ kvb.T)
    p = _bf16(np.exp(lg - lg.max(axis=1, keepdims=True)))
    o = (p @ kvb[:, :512]) / p.sum(axis=1, keepdims=True)
    mx, mean = _err(o, o_ref)
    assert mx < SFA_MAX_ABS / 4 and mean < SFA_MEAN_ABS / 4, (mx, mean)
