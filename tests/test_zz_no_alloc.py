"""The allocation-free Sparse Flash Attention entry point (dsa_sparse_attn_noalloc).

It exists for callers that cannot allocate device memory for the split-merge workspace
(a framework that owns every allocation, or a path where an allocation would synchronise
the device); it keeps that workspace in a fixed array inside the library.  Its output
must match dsa_sparse_attn with a caller-allocated workspace, call after call: the fixed
array keeps the previous call's contents, and those must not leak into the next result.

This file is collected last so that a run stopping at the first failure has already run
every other test.
"""

import numpy as np
import pytest
import torch

from dsa_sparse_attention_topk_gb300 import workloads as W
from dsa_testlib import ensure_built, DeviceWorkload, check_sfa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    return ensure_built()


def _both(dsa, dw, idx):
    wl = dw.wl
    ref_lse = torch.empty(wl.n_q, wl.h_s, dtype=torch.float32, device="cuda")
    ref, _ = dsa.sparse_attn(dw.q_sfa, dw.kv_cache, dw.page_table, dw.seq_lens, dw.q_seq, idx, wl.sm_scale,
                             out_lse=ref_lse)
    lse = torch.empty_like(ref_lse)
    out, _ = dsa.sparse_attn_noalloc(dw.q_sfa, dw.kv_cache, dw.page_table, dw.seq_lens, dw.q_seq, idx,
                                     wl.sm_scale, out_lse=lse)
    assert dsa.device_status() == 0
    return ref, ref_lse, out, lse


def _compare(ref, ref_lse, out, lse):
    check_sfa(out.float().cpu().numpy(), ref.float().cpu().numpy().astype(np.float64))
    fin = torch.isfinite(ref_lse)
    assert torch.equal(fin, torch.isfinite(lse))
    assert torch.allclose(lse[fin], ref_lse[fin], rtol=0, atol=1e-4)


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row(dsa):
    # three query rows: each row is split over several CTAs, so the scratch array is used
    wl = W.custom([3000, 1500, 700], h_i=16, h_s=128, topk=512, seed=41)
    assert dsa.sparse_attn_workspace_size(wl.n_q, wl.h_s, wl.topk) > 0
    dw = DeviceWorkload(wl)
    idx, _ = dw.indexer_topk(with_scores=False)
    for _ in range(2):
        _compare(*_both(dsa, dw, idx))


def test_noalloc_after_a_call_of_another_shape(dsa):
    # the previous contents of the shared array come from a different shape
    first = W.custom([2100, 900], h_i=16, h_s=64, topk=256, seed=42)
    second = W.custom([1200, 400, 2600, 64], h_i=16, h_s=128, topk=1024, seed=43)
    for wl in (first, second):
        dw = DeviceWorkload(wl)
        idx, _ = dw.indexer_topk(with_scores=False)
        _compare(*_both(dsa, dw, idx))


def test_noalloc_at_the_largest_split_layout(dsa):
    # nine rows of 2048 selected entries with 128 heads: the split count is as large as the
    # GPU allows for nine rows, and the workspace it needs must fit the fixed array
    wl = W.custom([2600 + 97 * i for i in range(9)], h_i=16, h_s=128, topk=2048, seed=44)
    need = dsa.sparse_attn_workspace_size(wl.n_q, wl.h_s, wl.topk)
    assert 0 < need <= dsa.NOALLOC_SCRATCH_BYTES
    dw = DeviceWorkload(wl)
    idx, _ = dw.indexer_topk(with_scores=False)
    ref, ref_lse, out, lse = _both(dsa, dw, idx)
    # the same kernels with the same split plan: equal bit for bit
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
