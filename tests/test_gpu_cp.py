"""Context-parallel decoding on the GPU.

* dsa_topk_merge against a plain stable sort of the candidates (score descending, then
  position ascending), with empty slots, ties across parts and NaN scores;
* dsa_lse_combine against the log-sum-exp weighting written out in numpy;
* the whole one-exchange flow with W = 2 and 4 ranks emulated as host threads on one GPU
  (each thread launches its rank's kernels; the exchange is a host-side all-gather, so no
  kernel ever waits for another), contiguous and zigzag shards: the merged Top-K must be
  the single-GPU Top-K set and the output must meet the attention tolerance against the
  oracle on that set.
"""

import threading

import numpy as np
import pytest
import torch

from dsa_sparse_attention_topk_gb300 import cp
from dsa_sparse_attention_topk_gb300 import workloads as W
from dsa_testlib import ensure_built, DeviceWorkload, OracleRows, check_sfa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    return ensure_built()


def _merge_ref(idx, sc, off, topk):
    P, n_q, K = idx.shape
    out = np.full((n_q, topk), -1, np.int64)
    for t in range(n_q):
        pos = (idx[:, t] + off[:, t, None]).reshape(-1)
        s = sc[:, t].reshape(-1).astype(np.float64)
        keep = idx[:, t].reshape(-1) >= 0
        pos, s = pos[keep], s[keep]
        nan = np.isnan(s)                       # NaN ranks below every other score
        order = np.lexsort((pos, -np.where(nan, 0, s), nan))[:topk]
        out[t, :order.size] = pos[order]
    return out


def test_topk_merge_matches_a_stable_sort(dsa):
    rng = np.random.default_rng(3)
    P, n_q, K, topk = 3, 5, 300, 257
    idx = rng.integers(0, 5000, size=(P, n_q, K)).astype(np.int32)
    sc = rng.integers(-40, 40, size=(P, n_q, K)).astype(np.float32) / 4   # many exact ties
    idx[0, 1, 100:] = -1                                                  # empty slots
    idx[:, 2, :] = -1
    idx[1, 2, :5] = [7, 8, 9, 10, 11]                                     # fewer than topk in all
    sc[2, 3, :10] = np.nan
    for t in range(n_q):                                                  # positions unique per row
        flat = idx[:, t].reshape(-1)
        live = flat >= 0
        flat[live] = rng.permutation(100000)[:live.sum()]
        idx[:, t] = flat.reshape(P, K)
    off = rng.integers(0, 1000, size=(P, n_q)).astype(np.int32)
    ci, cs, co = (torch.from_numpy(x).cuda() for x in (idx, sc, off))
    out, scores, _ = dsa.topk_merge(ci, cs, topk, part_offsets=co)
    assert dsa.device_status() == 0
    ref = _merge_ref(idx.astype(np.int64), sc, off.astype(np.int64), topk)
    assert np.array_equal(out.cpu().numpy(), ref)
    got = scores.cpu().numpy()
    assert np.all(np.isneginf(got[ref < 0]))


def test_topk_merge_local_selection(dsa):
    idx = torch.tensor([[[0, 5, 9, -1]], [[3, 1, 2, 0]]], dtype=torch.int32, device="cuda")  # 2 parts, 1 row
    sc = torch.tensor([[[1.0, 4.0, 2.0, 9.0]], [[3.0, 5.0, 0.5, 4.0]]], device="cuda")
    off = torch.tensor([[0], [10]], dtype=torch.int32, device="cuda")
    lo = torch.tensor([10], dtype=torch.int32, device="cuda")
    hi = torch.tensor([20], dtype=torch.int32, device="cuda")
    out, _, mine = dsa.topk_merge(idx, sc, 5, part_offsets=off, local_lo=lo, local_hi=hi)
    # by score: 11 (5), 5 (4), 10 (4: tie with 5, higher position), 13 (3), 9 (2)
    assert out.tolist() == [[11, 5, 10, 13, 9]]
    assert mine.tolist() == [[1, -1, 0, 3, -1]]


def test_lse_combine_matches_numpy(dsa):
    rng = np.random.default_rng(4)
    P, n_q, h = 3, 4, 16
    o = rng.standard_normal((P, n_q, h, 512)).astype(np.float32)
    lse = (rng.standard_normal((P, n_q, h)) * 3).astype(np.float32)
    lse[1, 2, :] = -np.inf                                # an empty part
    lse[:, 3, 5] = -np.inf                                # a head empty everywhere
    ob = torch.from_numpy(o).to(torch.bfloat16)
    out, out_lse = dsa.lse_combine(ob.cuda(), torch.from_numpy(lse).cuda())
    o64 = ob.double().numpy()
    L = np.logaddexp.reduce(lse.astype(np.float64), axis=0)
    with np.errstate(invalid="ignore"):
        w = np.where(np.isneginf(lse), 0.0, np.exp(lse - L))
    ref = np.nan_to_num((w[..., None] * o64).sum(0))
    assert np.abs(out.double().cpu().numpy() - ref).max() < 2e-2
    got = out_lse.cpu().numpy()
    assert np.allclose(got[np.isfinite(L)], L[np.isfinite(L)], atol=1e-5)
    assert np.all(np.isneginf(got[~np.isfinite(L)]))
    assert not out[3, 5].float().abs().sum().item()


class _Exchange:
    """A host-side all-gather between W threads (a barrier on each side)."""

    def __init__(self, world):
        self.world = world
        self.slots = [None] * world
        self.barrier = threading.Barrier(world)

    def for_rank(self, rank):
        def all_gather(t):
            self.slots[rank] = t
            self.barrier.wait()
            out = torch.stack(list(self.slots))
            self.barrier.wait()
            return out
        return all_gather


@pytest.mark.parametrize("world,zigzag", [(2, False), (2, True), (4, False)])
def test_context_parallel_flow_equals_the_single_gpu_path(dsa, world, zigzag):
    wl = W.custom([9000, 5000], per_seq=2, h_i=16, h_s=32, topk=512, seed=71)
    dw = DeviceWorkload(wl)
    ref_idx, _ = dw.indexer_topk(with_scores=False)
    ex = _Exchange(world)
    results, errors = {}, []

    def run(rank):
        try:
            views = cp.shard_views(torch.from_numpy(wl.page_table), torch.from_numpy(wl.seq_lens),
                                   torch.from_numpy(wl.q_seq), torch.from_numpy(wl.q_pos), world, rank, zigzag)
            be = cp.KernelBackend(dsa, dw.q_idx, dw.w, dw.q_sfa, dw.k_cache, dw.kv_cache, wl.sm_scale,
                                  ex.for_rank(rank), q_group=wl.q_group)
            results[rank] = cp.cp_decode(be, views, wl.topk)
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)
            ex.barrier.abort()

    threads = [threading.Thread(target=run, args=(r,)) for r in range(world)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not errors, errors
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    ref_sets = [set(r[r >= 0].tolist()) for r in ref_idx.cpu().numpy()]
    orc = OracleRows(wl)
    qs = wl.q_sfa().double().numpy()
    out0 = results[0][0]
    for rank in range(world):
        out, lse, idx = results[rank]
        idx = idx.cpu().numpy()
        for t in range(wl.n_q):
            assert set(idx[t][idx[t] >= 0].tolist()) == ref_sets[t]
        assert torch.equal(out, out0)                 # every rank holds the same result
    idx0 = results[0][2].cpu().numpy()
    for t in range(wl.n_q):
        o_ref, _ = orc.sfa(t, idx0[t], qs[t])
        check_sfa(out0[t].float().cpu().numpy(), o_ref)
