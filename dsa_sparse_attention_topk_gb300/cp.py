"""Context-parallel decoding: the one-exchange split of one long context over W devices.

"Deep Dive into Sparse Attention and Engineering Optimizations for Efficient Inference in
Kimi K3.1 Pro", section 3 ("Introduction of Context Parallelism"), and "Adapting and
Optimizing Kimi K3.1 Pro for Long-Sequence Inference", section 4: the context of a long
sequence is sharded over the devices.  Each device

1. runs the fused indexer + Top-K over its own shard, keeping K local candidates with
   their scores;
2. exchanges those candidates once (all-gather) and merges them into the global Top-K,
   identical on every device;
3. runs sparse attention over the selected entries that lie in its shard;
4. exchanges (o, lse) once more and combines them with log-sum-exp weights.

The result equals the single-device path: the merged Top-K is the Top-K of all scores,
and softmax attention over a union of disjoint entry sets is the log-sum-exp weighting of
the attentions over the sets.  "Kimi K3.1 Pro Inference Acceleration ...", section "Zigzag
Layout: Balancing Cross-Card Indexing Compute Load", pairs an early and a late chunk on
every device so that causal prefill rows cost every device about the same
(``zigzag=True``).

This module only plans the shards (page-aligned position ranges, page-table slices and
position offsets) and orders the calls; every computation is a call of the backend, which
for a GPU is :class:`KernelBackend` (the library's kernels) and whose ``all_gather`` is
the exchange (for instance ``torch.distributed.all_gather``).
"""

from dataclasses import dataclass

import torch

PAGE = 64


def plan_chunks(seq_len, world, rank, zigzag=False):
    """Position ranges [lo, hi) of one sequence that ``rank`` holds: one contiguous
    page-aligned range, or (zigzag) chunks r and 2W-1-r of 2W page-aligned chunks."""
    n_pages = (int(seq_len) + PAGE - 1) // PAGE
    parts = 2 * world if zigzag else world
    cuts = [n_pages * i // parts for i in range(parts + 1)]
    mine = [rank, 2 * world - 1 - rank] if zigzag else [rank]
    out = []
    for c in sorted(mine):
        lo, hi = cuts[c] * PAGE, min(cuts[c + 1] * PAGE, int(seq_len))
        out.append((lo, max(lo, hi)))
    return out


@dataclass
class ShardView:
    """One chunk of every sequence seen as sequences of their own: the page-table slices,
    the chunk lengths, the query positions relative to each chunk's first position, and
    per query row the chunk's global range [lo, hi)."""
    page_table: torch.Tensor   # int32 [B, max_pages_local]
    seq_lens: torch.Tensor     # int32 [B]
    q_seq: torch.Tensor        # int32 [n_q]
    q_pos: torch.Tensor        # int32 [n_q] (negative: the row selects nothing here)
    row_lo: torch.Tensor       # int32 [n_q]
    row_hi: torch.Tensor       # int32 [n_q]
    max_ctx: int


def shard_views(page_table, seq_lens, q_seq, q_pos, world, rank, zigzag=False):
    """The views of ``rank``'s chunks (one, or two with zigzag), built from host (CPU)
    int32 tensors; the caller moves them to its device."""
    page_table = page_table.cpu()
    seq_lens = [int(x) for x in seq_lens.cpu().tolist()]
    q_seq_l = [int(x) for x in q_seq.cpu().tolist()]
    q_pos_l = [int(x) for x in q_pos.cpu().tolist()]
    per_seq = [plan_chunks(L, world, rank, zigzag) for L in seq_lens]
    n_chunks = len(per_seq[0]) if per_seq else (2 if zigzag else 1)
    views = []
    for c in range(n_chunks):
        ranges = [chunks[c] for chunks in per_seq]
        lens = [hi - lo for lo, hi in ranges]
        max_len = max(lens + [1])
        max_pages = max(1, (max_len + PAGE - 1) // PAGE)
        pt = torch.full((len(seq_lens), max_pages), -1, dtype=torch.int32)
        for b, (lo, hi) in enumerate(ranges):
            n = (hi - lo + PAGE - 1) // PAGE
            if n:
                pt[b, :n] = page_table[b, lo // PAGE:lo // PAGE + n]
        row_lo = torch.tensor([ranges[s][0] for s in q_seq_l], dtype=torch.int32)
        row_hi = torch.tensor([ranges[s][1] for s in q_seq_l], dtype=torch.int32)
        views.append(ShardView(pt, torch.tensor(lens, dtype=torch.int32), torch.tensor(q_seq_l, dtype=torch.int32),
                               torch.tensor([p - ranges[s][0] for p, s in zip(q_pos_l, q_seq_l)], dtype=torch.int32),
                               row_lo, row_hi, max_pages * PAGE))
    return views


def cp_decode(backend, views, topk):
    """One context-parallel decode step of this device over its chunk views.  Returns
    (out [n_q, h, 512], lse [n_q, h], idx [n_q, topk]); every device gets the same."""
    # 1. local candidates of every chunk this device holds
    local = [backend.indexer_topk(v, topk) for v in views]
    cand_idx = torch.stack([c[0] for c in local])          # [chunks, n_q, K]
    cand_scores = torch.stack([c[1] for c in local])
    offsets = torch.stack([v.row_lo for v in views]).to(cand_idx.device)
    # 2. the first exchange, then the merge (the local selections come with it)
    all_idx = backend.all_gather(cand_idx).flatten(0, 1)   # [W * chunks, n_q, K]
    all_scores = backend.all_gather(cand_scores).flatten(0, 1)
    all_offsets = backend.all_gather(offsets).flatten(0, 1)
    idx, mine = None, []
    for v in views:
        idx, sel = backend.topk_merge(all_idx, all_scores, all_offsets, topk, v.row_lo, v.row_hi)
        mine.append(sel)
    # 3. attention over the selected entries this device holds
    parts = [backend.sparse_attn(v, sel) for v, sel in zip(views, mine)]
    o = torch.stack([p[0] for p in parts])                  # [chunks, n_q, h, 512]
    lse = torch.stack([p[1] for p in parts])
    # 4. the second exchange and the log-sum-exp combination
    out, out_lse = backend.lse_combine(backend.all_gather(o).flatten(0, 1), backend.all_gather(lse).flatten(0, 1))
    return out, out_lse, idx


class KernelBackend:
    """The library's kernels on one GPU.  ``all_gather`` stacks a tensor of every device
    along a new first dimension (``torch.distributed`` over NCCL, or any other
    exchange)."""

    def __init__(self, dsa, q_idx, w, q_sfa, k_cache, kv_cache, sm_scale, all_gather, q_group=1):
        self.dsa, self.q_idx, self.w, self.q_sfa = dsa, q_idx, w, q_sfa
        self.k_cache, self.kv_cache, self.sm_scale = k_cache, kv_cache, sm_scale
        self.q_group = q_group
        self._gather = all_gather

    def _dev(self, v):
        d = self.q_idx.device
        return (v.page_table.to(d), v.seq_lens.to(d), v.q_seq.to(d), v.q_pos.to(d))

    def indexer_topk(self, v, topk):
        pt, sl, qs, qp = self._dev(v)
        sc = torch.empty(qs.shape[0], topk, dtype=torch.float32, device=self.q_idx.device)
        idx, sc = self.dsa.indexer_topk(self.q_idx, self.w, self.k_cache, pt, sl, qs, qp, topk, v.max_ctx,
                                        q_group=self.q_group, out_scores=sc)
        return idx, sc

    def all_gather(self, t):
        return self._gather(t)

    def topk_merge(self, cand_idx, cand_scores, offsets, topk, lo, hi):
        d = self.q_idx.device
        idx, _, sel = self.dsa.topk_merge(cand_idx.contiguous(), cand_scores.contiguous(), topk,
                                          part_offsets=offsets.to(d).contiguous(), local_lo=lo.to(d),
                                          local_hi=hi.to(d))
        return idx, sel

    def sparse_attn(self, v, sel):
        pt, sl, qs, _ = self._dev(v)
        lse = torch.empty(qs.shape[0], self.q_sfa.shape[1], dtype=torch.float32, device=self.q_idx.device)
        out, lse = self.dsa.sparse_attn(self.q_sfa, self.kv_cache, pt, sl, qs, sel, self.sm_scale, out_lse=lse)
        return out, lse

    def lse_combine(self, o_parts, lse_parts):
        return self.dsa.lse_combine(o_parts.contiguous(), lse_parts.contiguous())
