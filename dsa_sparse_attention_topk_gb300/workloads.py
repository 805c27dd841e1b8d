"""Seeded synthetic inputs for the DSA decode path.

This module only draws random numbers and lays out pages; it holds none of the method's
arithmetic (no quantisation, scoring, selection or attention), so the CPU oracle and the
CUDA path can both be fed from it without sharing any of the computation.

Every tensor of a workload comes from its own counter-keyed numpy PCG64 stream,
``SeedSequence([seed, tag, index])``, so any single sequence can be regenerated alone
(the oracle recomputes sampled rows without drawing the whole batch).  Values are drawn
in float32 and rounded to bfloat16 by torch (round to nearest even).

The five named workloads (their shapes, value distributions and structure):

1. ``tiny``: 1 sequence of 4096 tokens, 1 query row; indexer 8 heads x 128, w ~ N(0, 1/8);
   Top-K 256; SFA 16 heads x 576; seed 0.
2. ``decode_b32_ctx32k``: 32 sequences x 32768 tokens, 1 query row each; indexer 64 x 128,
   w ~ N(0, 1/64), 4 seeded outlier channels of indexer q and k scaled by 8; Top-K 2048;
   SFA 128 x 576; seed 1.
3. ``mixed_b128``: 128 sequences, lengths log-uniform over [4096, 131072]; one query row
   each; Top-K 2048 (all positions when fewer); seed 2.
4. ``long_mtp_b4_ctx128k``: 4 sequences x 131072 tokens, 2 query rows each at positions
   L-2 and L-1; 1% of keys planted with cosine 0.5 to the first row's weighted query;
   seed 3.
5. ``prefill_4k_over_64k``: 1 sequence of 65536 tokens, 4096 query rows at positions
   61440..65535 (causal); seed 4.

plus ``short_ctx`` (2 sequences of 1000 and 64 tokens, Top-K 2048: fewer selectable
positions than K; seed 5).  In all of them q, k and the latent kv are N(0, 1) before the
bfloat16 rounding, the page size is 64, and physical pages are a seeded permutation of
one shared pool.
"""

from dataclasses import dataclass, field
import math

import numpy as np
import torch

PAGE = 64
D_INDEX = 128
D_LATENT = 576
D_V = 512

# stream tags
_T_K, _T_KV, _T_QI, _T_W, _T_QS, _T_LEN, _T_PERM, _T_OUTLIER, _T_PLANT = range(1, 10)


def _rng(seed, tag, index=0):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), tag, int(index)])))


def _bf16(a):
    """float32/float64 numpy -> torch.bfloat16 (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


@dataclass
class Workload:
    name: str
    seed: int
    seq_lens: np.ndarray          # int32 [B]
    q_seq: np.ndarray             # int32 [NQ] sequence of each query row
    q_pos: np.ndarray             # int32 [NQ] position of each query row
    q_group: int                  # consecutive query rows sharing one sequence
    h_i: int
    h_s: int
    topk: int
    w_std: float
    outliers: int = 0             # number of indexer channels scaled by 8
    planted_frac: float = 0.0     # fraction of keys planted towards the query
    sm_scale: float = 1.0 / math.sqrt(192.0)
    page_table: np.ndarray = field(default=None)   # int32 [B, max_pages], -1 = unused
    num_pages: int = 0

    # ---- layout -------------------------------------------------------------------
    def __post_init__(self):
        self.seq_lens = np.asarray(self.seq_lens, dtype=np.int32)
        self.q_seq = np.asarray(self.q_seq, dtype=np.int32)
        self.q_pos = np.asarray(self.q_pos, dtype=np.int32)
        if self.page_table is None:
            n_pages = [(int(L) + PAGE - 1) // PAGE for L in self.seq_lens]
            self.num_pages = int(sum(n_pages))
            perm = _rng(self.seed, _T_PERM).permutation(self.num_pages).astype(np.int32)
            maxp = max(n_pages) if n_pages else 0
            pt = np.full((len(n_pages), maxp), -1, dtype=np.int32)
            off = 0
            for b, n in enumerate(n_pages):
                pt[b, :n] = perm[off:off + n]
                off += n
            self.page_table = pt

    @property
    def B(self):
        return int(self.seq_lens.shape[0])

    @property
    def n_q(self):
        return int(self.q_seq.shape[0])

    @property
    def max_pages(self):
        return int(self.page_table.shape[1])

    @property
    def max_ctx(self):
        return int(self.seq_lens.max()) if self.B else 0

    @property
    def num_slots(self):
        return self.num_pages * PAGE

    def identity_pages(self):
        """The same workload with pages laid out in order (page table = 0, 1, 2, ...)."""
        pt = np.full_like(self.page_table, -1)
        off = 0
        for b, L in enumerate(self.seq_lens):
            n = (int(L) + PAGE - 1) // PAGE
            pt[b, :n] = np.arange(off, off + n, dtype=np.int32)
            off += n
        w = Workload(self.name + "_identity", self.seed, self.seq_lens, self.q_seq, self.q_pos,
                     self.q_group, self.h_i, self.h_s, self.topk, self.w_std, self.outliers,
                     self.planted_frac, self.sm_scale, pt, self.num_pages)
        return w

    def slot_mapping(self, b):
        """int64 [ctx_b]: cache slot (physical page * 64 + offset) of every token of seq b."""
        L = int(self.seq_lens[b])
        p = np.arange(L)
        return (self.page_table[b, p // PAGE].astype(np.int64) * PAGE + (p % PAGE)).astype(np.int64)

    # ---- values -------------------------------------------------------------------
    def _outlier_channels(self):
        if not self.outliers:
            return None
        return _rng(self.seed, _T_OUTLIER).choice(D_INDEX, size=self.outliers, replace=False)

    def q_index(self):
        """bf16 [NQ, H_I, 128] indexer queries (outlier channels already scaled)."""
        q = _rng(self.seed, _T_QI).standard_normal((self.n_q, self.h_i, D_INDEX), dtype=np.float32)
        ch = self._outlier_channels()
        qb = _bf16(q)
        if ch is not None:
            qb[:, :, torch.from_numpy(ch)] *= 8  # exact in bf16
        return qb

    def weights(self):
        """fp32 [NQ, H_I] head weights, N(0, w_std^2)."""
        w = _rng(self.seed, _T_W).standard_normal((self.n_q, self.h_i), dtype=np.float32)
        return torch.from_numpy(w * np.float32(self.w_std))

    def q_sfa(self, rows=None):
        """bf16 [NQ, H_S, 576] absorbed MLA queries (or only the given rows)."""
        rows = range(self.n_q) if rows is None else rows
        out = []
        for r in rows:
            q = _rng(self.seed, _T_QS, r).standard_normal((self.h_s, D_LATENT), dtype=np.float32)
            out.append(_bf16(q))
        return torch.stack(out) if out else torch.empty(0, self.h_s, D_LATENT, dtype=torch.bfloat16)

    def k_seq(self, b, q_index=None, weights=None):
        """bf16 [ctx_b, 128] indexer keys of sequence b (outliers and planted keys applied)."""
        L = int(self.seq_lens[b])
        k = _rng(self.seed, _T_K, b).standard_normal((L, D_INDEX), dtype=np.float32)
        if self.planted_frac > 0:
            qi = self.q_index() if q_index is None else q_index
            ww = self.weights() if weights is None else weights
            t0 = int(np.nonzero(self.q_seq == b)[0][0])
            u = (ww[t0].double()[:, None] * qi[t0].double()).sum(0).numpy()
            u = u / np.linalg.norm(u)
            g_rng = _rng(self.seed, _T_PLANT, b)
            n_plant = int(round(self.planted_frac * L))
            pos = g_rng.choice(L, size=n_plant, replace=False)
            g = g_rng.standard_normal((n_plant, D_INDEX))
            vperp = g - (g @ u)[:, None] * u[None, :]
            vperp /= np.linalg.norm(vperp, axis=1, keepdims=True)
            k[pos] = (np.linalg.norm(g, axis=1, keepdims=True)
                      * (0.5 * u[None, :] + math.sqrt(0.75) * vperp)).astype(np.float32)
        kb = _bf16(k)
        ch = self._outlier_channels()
        if ch is not None:
            kb[:, torch.from_numpy(ch)] *= 8
        return kb

    def kv_seq(self, b):
        """bf16 [ctx_b, 576] MLA latent rows (512 nope + 64 rope) of sequence b."""
        L = int(self.seq_lens[b])
        kv = _rng(self.seed, _T_KV, b).standard_normal((L, D_LATENT), dtype=np.float32)
        return _bf16(kv)

    def seq_rows(self, b):
        return np.nonzero(self.q_seq == b)[0]


def _decode_rows(seq_lens, per_seq):
    q_seq, q_pos = [], []
    for b, L in enumerate(seq_lens):
        for j in range(per_seq):
            q_seq.append(b)
            q_pos.append(int(L) - per_seq + j)
    return np.array(q_seq, np.int32), np.array(q_pos, np.int32)


def make(name):
    """One of the named workloads (see the module docstring)."""
    if name == "tiny":
        L = np.array([4096])
        qs, qp = _decode_rows(L, 1)
        return Workload(name, 0, L, qs, qp, 1, h_i=8, h_s=16, topk=256, w_std=math.sqrt(1 / 8))
    if name == "decode_b32_ctx32k":
        L = np.full(32, 32768)
        qs, qp = _decode_rows(L, 1)
        return Workload(name, 1, L, qs, qp, 1, h_i=64, h_s=128, topk=2048, w_std=1 / 8, outliers=4)
    if name == "mixed_b128":
        u = _rng(2, _T_LEN).uniform(math.log(4096), math.log(131072), size=128)
        L = np.clip(np.floor(np.exp(u)), 4096, 131072).astype(np.int32)
        qs, qp = _decode_rows(L, 1)
        return Workload(name, 2, L, qs, qp, 1, h_i=64, h_s=128, topk=2048, w_std=1 / 8)
    if name == "long_mtp_b4_ctx128k":
        L = np.full(4, 131072)
        qs, qp = _decode_rows(L, 2)
        return Workload(name, 3, L, qs, qp, 2, h_i=64, h_s=128, topk=2048, w_std=1 / 8,
                        planted_frac=0.01)
    if name == "prefill_4k_over_64k":
        L = np.array([65536])
        qp = np.arange(61440, 65536, dtype=np.int32)
        qs = np.zeros(4096, np.int32)
        return Workload(name, 4, L, qs, qp, 4, h_i=64, h_s=128, topk=2048, w_std=1 / 8)
    if name == "short_ctx":
        L = np.array([1000, 64])
        qs, qp = _decode_rows(L, 1)
        return Workload(name, 5, L, qs, qp, 1, h_i=64, h_s=128, topk=2048, w_std=1 / 8)
    raise KeyError(name)


def custom(seq_lens, per_seq=1, h_i=64, h_s=128, topk=2048, seed=11, outliers=0,
           planted_frac=0.0, name="custom"):
    """A decode workload of arbitrary sequence lengths (for ragged and edge cases)."""
    L = np.asarray(seq_lens, np.int32)
    qs, qp = _decode_rows(L, per_seq)
    return Workload(name, seed, L, qs, qp, per_seq, h_i=h_i, h_s=h_s, topk=topk,
                    w_std=1 / math.sqrt(h_i), outliers=outliers, planted_frac=planted_frac)


NAMES = ["tiny", "decode_b32_ctx32k", "mixed_b128", "long_mtp_b4_ctx128k",
         "prefill_4k_over_64k", "short_ctx"]
