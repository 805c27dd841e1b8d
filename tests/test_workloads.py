"""Host checks of the seeded input generators: determinism, page layout, outliers,
planted keys and the query-row layout of every named workload."""

import ast
import os

import numpy as np
import torch

from dsa_sparse_attention_topk_gb300 import workloads as W

PKG = os.path.join(os.path.dirname(os.path.dirname(__file__)), "dsa_sparse_attention_topk_gb300")


def test_generator_module_holds_no_oracle_import():
    tree = ast.parse(open(os.path.join(PKG, "workloads.py")).read())
    names = [n.module or "" for n in ast.walk(tree) if isinstance(n, ast.ImportFrom)]
    names += [a.name for n in ast.walk(tree) if isinstance(n, ast.Import) for a in n.names]
    assert not any("oracle" in n for n in names)


def test_named_shapes():
    t = W.make("tiny")
    assert (t.B, t.n_q, t.h_i, t.h_s, t.topk) == (1, 1, 8, 16, 256)
    assert t.q_pos.tolist() == [4095]
    d = W.make("decode_b32_ctx32k")
    assert (d.B, d.n_q, d.h_i, d.h_s, d.topk, d.max_ctx) == (32, 32, 64, 128, 2048, 32768)
    m = W.make("mixed_b128")
    assert m.B == 128 and m.seq_lens.min() >= 4096 and m.seq_lens.max() <= 131072
    lm = W.make("long_mtp_b4_ctx128k")
    assert lm.n_q == 8 and lm.q_group == 2 and lm.q_pos.tolist()[:2] == [131070, 131071]
    p = W.make("prefill_4k_over_64k")
    assert p.n_q == 4096 and p.q_pos[0] == 61440 and p.q_pos[-1] == 65535
    s = W.make("short_ctx")
    assert s.seq_lens.tolist() == [1000, 64]


def test_page_table_is_a_permutation_and_slots_match():
    w = W.custom([130, 64, 1, 700], seed=3)
    used = np.concatenate([w.page_table[b, :(int(L) + 63) // 64] for b, L in enumerate(w.seq_lens)])
    assert sorted(used.tolist()) == list(range(w.num_pages))
    assert np.all(w.page_table[0, 3:] == -1)
    sm = w.slot_mapping(3)
    assert sm.shape == (700,) and sm[65] == w.page_table[3, 1] * 64 + 1
    ident = w.identity_pages()
    assert ident.slot_mapping(0).tolist() == list(range(130))


def test_determinism_and_independent_streams():
    a = W.custom([100, 50], seed=9)
    b = W.custom([100, 50], seed=9)
    assert torch.equal(a.k_seq(1), b.k_seq(1)) and torch.equal(a.kv_seq(0), b.kv_seq(0))
    assert torch.equal(a.q_sfa([1])[0], a.q_sfa()[1])
    assert not torch.equal(a.k_seq(0)[:50], a.k_seq(1))


def test_outlier_channels_scaled_by_8():
    w = W.custom([64], outliers=4, seed=2)
    base = W.custom([64], outliers=0, seed=2)
    k, k0 = w.k_seq(0).double(), base.k_seq(0).double()
    ratio = (k / k0.where(k0 != 0, torch.ones_like(k0)))
    cols = [c for c in range(128) if torch.all((ratio[:, c] == 8) | (k0[:, c] == 0))]
    assert len(cols) == 4
    q, q0 = w.q_index().double(), base.q_index().double()
    assert torch.equal(q[..., cols], q0[..., cols] * 8)


def test_planted_keys_have_cosine_half():
    w = W.custom([2000], h_i=8, planted_frac=0.01, seed=4)
    k = w.k_seq(0).double().numpy()
    u = (w.weights()[0].double()[:, None] * w.q_index()[0].double()).sum(0).numpy()
    u /= np.linalg.norm(u)
    cos = (k @ u) / np.linalg.norm(k, axis=1)
    planted = np.abs(cos - 0.5) < 0.02
    assert planted.sum() >= 20                 # 1% of 2000 (bf16 rounding moves cos a little)
    assert np.sum(cos > 0.45) <= 20 + 2        # random N(0, I) keys almost never reach 0.45
