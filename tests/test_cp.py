"""Context-parallel decoding on the CPU: the shard plan, the log-sum-exp identity the
combination step rests on, and the whole one-exchange flow over two gloo ranks with the
float64 oracle standing in for the kernels.  The flow must give exactly the oracle's
single-device Top-K and its attention output ("Deep Dive into Sparse Attention ...",
section 3; "Adapting and Optimizing Kimi K3.1 Pro for Long-Sequence Inference", section 4).
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from dsa_sparse_attention_topk_gb300 import cp
from dsa_sparse_attention_topk_gb300 import workloads as W


@pytest.mark.parametrize("zigzag", [False, True])
@pytest.mark.parametrize("world", [1, 2, 3, 4])
@pytest.mark.parametrize("L", [1, 63, 64, 1000, 4097])
def test_plan_covers_the_context_once(world, zigzag, L):
    seen = []
    for r in range(world):
        chunks = cp.plan_chunks(L, world, r, zigzag)
        assert len(chunks) == (2 if zigzag else 1)
        for lo, hi in chunks:
            assert lo % cp.PAGE == 0 and lo <= hi <= L
            seen.extend(range(lo, hi))
    assert sorted(seen) == list(range(L))


def test_zigzag_pairs_an_early_and_a_late_chunk():
    # 8 chunks over 4 ranks: rank r holds chunks r and 7 - r
    L = 8 * 640
    assert cp.plan_chunks(L, 4, 0, True) == [(0, 640), (7 * 640, 8 * 640)]
    assert cp.plan_chunks(L, 4, 3, True) == [(3 * 640, 4 * 640), (4 * 640, 5 * 640)]


def test_attention_over_a_union_is_the_lse_weighting_of_the_parts():
    rng = np.random.default_rng(11)
    q = rng.standard_normal((4, 576))
    kv = rng.standard_normal((50, 576))
    idx = rng.permutation(50)
    parts = [idx[:20], idx[20:21], idx[21:]]
    o_ref, lse_ref = oracle.sparse_attention_row(q, kv, idx, 0.07)
    os_, ls = zip(*[oracle.sparse_attention_row(q, kv, p, 0.07) for p in parts])
    L = np.logaddexp.reduce(np.stack(ls), axis=0)
    o = sum(np.exp(l - L)[:, None] * o_p for o_p, l in zip(os_, ls))
    assert np.allclose(o, o_ref, rtol=0, atol=1e-13) and np.allclose(L, lse_ref, rtol=0, atol=1e-13)


# ---- the whole flow over gloo ranks, with the oracle standing in for the kernels -------

class OracleBackend:
    """float64 stand-ins for the library's calls, over logical (unpaged) sequences."""

    def __init__(self, wl, all_gather):
        self.wl = wl
        self.gather = all_gather
        q = wl.q_index().double().numpy()
        self.q_hat = [oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(q[r])) for r in range(wl.n_q)]
        self.w = wl.weights().double().numpy()
        self.q_sfa = wl.q_sfa().double().numpy()
        self.k_hat = [oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(wl.k_seq(b).double().numpy()))
                      for b in range(wl.B)]
        self.kv_hat = [oracle.fp8_tile_dequantize(*oracle.fp8_tile_quantize(wl.kv_seq(b).double().numpy()))
                       for b in range(wl.B)]

    def all_gather(self, t):
        return self.gather(t)

    def indexer_topk(self, v, topk):
        idx = torch.full((self.wl.n_q, topk), -1, dtype=torch.int32)
        sc = torch.full((self.wl.n_q, topk), -np.inf, dtype=torch.float64)
        for t in range(self.wl.n_q):
            b, lo = int(v.q_seq[t]), int(v.row_lo[t])
            n = max(0, min(int(v.q_pos[t]) + 1, int(v.seq_lens[b])))
            s = oracle.indexer_scores_row(self.q_hat[t], self.w[t], self.k_hat[b][lo:lo + n])
            i, vals = oracle.topk_row(s, topk)
            idx[t] = torch.from_numpy(i)
            sc[t] = torch.from_numpy(vals)
        return idx, sc

    def topk_merge(self, cand_idx, cand_scores, offsets, topk, lo, hi):
        n_q = cand_idx.shape[1]
        out = torch.full((n_q, topk), -1, dtype=torch.int32)
        mine = torch.full((n_q, topk), -1, dtype=torch.int32)
        for t in range(n_q):
            pos = (cand_idx[:, t] + offsets[:, t, None]).flatten().numpy()
            s = cand_scores[:, t].flatten().numpy()
            keep = cand_idx[:, t].flatten().numpy() >= 0
            pos, s = pos[keep], s[keep]
            order = np.lexsort((pos, -s))[:topk]
            out[t, :order.size] = torch.from_numpy(pos[order].astype(np.int32))
            sel = out[t]
            inside = (sel >= lo[t]) & (sel < hi[t]) & (sel >= 0)
            mine[t] = torch.where(inside, sel - lo[t], torch.full_like(sel, -1))
        return out, mine

    def sparse_attn(self, v, sel):
        H = self.q_sfa.shape[1]
        o = torch.zeros(self.wl.n_q, H, 512, dtype=torch.float64)
        lse = torch.full((self.wl.n_q, H), -np.inf, dtype=torch.float64)
        for t in range(self.wl.n_q):
            b, lo, hi = int(v.q_seq[t]), int(v.row_lo[t]), int(v.row_hi[t])
            oo, ll = oracle.sparse_attention_row(self.q_sfa[t], self.kv_hat[b][lo:hi], sel[t].numpy(),
                                                 self.wl.sm_scale)
            o[t], lse[t] = torch.from_numpy(oo), torch.from_numpy(ll)
        return o, lse

    def lse_combine(self, o_parts, lse_parts):
        L = torch.logsumexp(lse_parts, dim=0)
        wgt = torch.where(torch.isneginf(lse_parts), torch.zeros_like(lse_parts), torch.exp(lse_parts - L))
        o = (wgt[..., None] * o_parts).sum(0)
        return torch.nan_to_num(o), L


def _workload():
    # two sequences with MTP rows: the second row of each pair attends causally to the first
    return W.custom([2300, 900], per_seq=2, h_i=8, h_s=8, topk=200, seed=61)


def _single_device_oracle(wl):
    orc = OracleBackend(wl, None)
    idx = np.full((wl.n_q, wl.topk), -1, np.int64)
    o = np.zeros((wl.n_q, wl.h_s, 512))
    for t in range(wl.n_q):
        b = int(wl.q_seq[t])
        n = oracle.indexer.selectable_count(wl.q_pos[t], wl.seq_lens[b])
        s = oracle.indexer_scores_row(orc.q_hat[t], orc.w[t], orc.k_hat[b][:n])
        idx[t], _ = oracle.topk_row(s, wl.topk)
        o[t], _ = oracle.sparse_attention_row(orc.q_sfa[t], orc.kv_hat[b], idx[t], wl.sm_scale)
    return idx, o


def _rank(rank, world, port, zigzag, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = _workload()

        def all_gather(t):
            bufs = [torch.empty_like(t) for _ in range(world)]
            dist.all_gather(bufs, t.contiguous())
            return torch.stack(bufs)

        views = cp.shard_views(torch.from_numpy(wl.page_table), torch.from_numpy(wl.seq_lens),
                               torch.from_numpy(wl.q_seq), torch.from_numpy(wl.q_pos), world, rank, zigzag)
        out, lse, idx = cp.cp_decode(OracleBackend(wl, all_gather), views, wl.topk)
        q.put((rank, idx.numpy(), out.numpy()))
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("zigzag", [False, True])
def test_two_gloo_ranks_equal_the_single_device_oracle(zigzag):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, zigzag, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl = _workload()
    idx_ref, o_ref = _single_device_oracle(wl)
    for rank, idx, out in res:
        assert np.array_equal(idx, idx_ref), f"rank {rank}: merged Top-K differs"
        assert np.allclose(out, o_ref, rtol=0, atol=1e-12)

