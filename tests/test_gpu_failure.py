"""Failure handling on the GPU, provoked without any fault:

* a bounded wait that runs out: the indexer's copy producer is stalled through the
  library's testing hook, so its consumers' waits give up after 2 ms; the call must come
  back with DSA_STATUS_TIMEOUT and rows of -1, and the next normal call must give the
  earlier result with a clean status word (the kernel freed its tensor memory and left
  nothing waiting);
* NaN scores: a NaN head weight makes every score of its row NaN; such scores rank below
  every other score (a stable descending sort puts NaN last), so the row keeps its K lowest
  positions, reports NaN scores and sets DSA_STATUS_NAN_SCORE, while the other rows are
  untouched;
* positions on pages flagged bad leave fewer than K selectable keys in a long row: the row
  keeps every valid position and is padded with -1.
"""

import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_topk_gb300 import workloads as W
from dsa_testlib import ensure_built, DeviceWorkload, OracleRows, check_topk

pytestmark = pytest.mark.gpu

TIMEOUT, BAD_PAGE, NAN_SCORE = 16, 1, 32


@pytest.fixture(scope="module")
def dsa():
    return ensure_built()


def _topk(dsa, dw, w=None, page_table=None):
    wl = dw.wl
    sc = torch.empty(wl.n_q, wl.topk, dtype=torch.float32, device="cuda")
    return dsa.indexer_topk(dw.q_idx, dw.w if w is None else w, dw.k_cache,
                            dw.page_table if page_table is None else page_table, dw.seq_lens, dw.q_seq,
                            dw.q_pos, wl.topk, wl.max_ctx, q_group=wl.q_group, out_scores=sc)


def test_stalled_producer_times_out_and_the_next_call_is_clean(dsa):
    wl = W.custom([3000, 2500, 5000], h_i=16, h_s=32, topk=256, seed=23)
    dw = DeviceWorkload(wl, with_kv=False)
    idx_ok, sc_ok = _topk(dsa, dw)
    assert dsa.device_status() == 0
    dsa.test_stall_indexer(2000)
    try:
        idx_bad, _ = _topk(dsa, dw)
        bits = dsa.device_status()
    finally:
        dsa.test_stall_indexer(0)
    assert bits & TIMEOUT, dsa.status_names(bits)
    assert torch.all(idx_bad == -1)
    idx2, sc2 = _topk(dsa, dw)
    assert dsa.device_status() == 0
    assert torch.equal(idx2, idx_ok) and torch.equal(sc2, sc_ok)


def test_stall_hook_rejects_bad_limits(dsa):
    with pytest.raises(dsa.DsaError):
        dsa.test_stall_indexer(-1)


def test_nan_scores_rank_last(dsa):
    wl = W.custom([700, 300], h_i=8, h_s=16, topk=64, seed=29)
    dw = DeviceWorkload(wl, with_kv=False)
    w = dw.w.clone()
    w[0, 3] = float("nan")
    idx, sc = _topk(dsa, dw, w=w)
    bits = dsa.device_status()
    assert bits == NAN_SCORE, dsa.status_names(bits)
    idx, sc = idx.cpu().numpy(), sc.cpu().numpy()
    orc = OracleRows(wl)
    orc.w[0] = w[0].double().cpu().numpy()
    ref_idx, s, mag = orc.topk(0)
    assert np.all(np.isnan(s))                        # the oracle's scores of row 0 are NaN too
    assert sorted(idx[0].tolist()) == sorted(ref_idx.tolist()) == list(range(wl.topk))
    assert np.all(np.isnan(sc[0]))
    ref_idx1, s1, mag1 = orc.topk(1)
    check_topk(idx[1], sc[1], s1, mag1, wl.topk)


def test_bad_pages_leave_fewer_than_k_and_pad(dsa):
    wl = W.custom([4000], h_i=16, h_s=32, topk=512, seed=31)
    dw = DeviceWorkload(wl, with_kv=False)
    pt = dw.page_table.clone()
    n_pages = (4000 + 63) // 64
    pt[0, 4:n_pages] = -7                              # only positions 0..255 stay valid
    idx, sc = _topk(dsa, dw, page_table=pt)
    bits = dsa.device_status()
    assert bits & BAD_PAGE
    idx = idx[0].cpu().numpy()
    assert sorted(idx[idx >= 0].tolist()) == list(range(256))
    assert np.all(idx[256:] == -1) and np.all(idx[:256] >= 0)   # valid positions first, then -1
