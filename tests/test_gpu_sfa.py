"""GPU parity of Sparse Flash Attention against the float64 oracle (max-abs 2e-2,
mean-abs 2e-3 on the bf16 output; lse within the bf16 rounding's worst case of the float64
oracle and within 1e-4 of the oracle over the bf16-rounded latent rows), fed with the
oracle's own Top-K indices, plus padding, empty rows, out-of-range indices and fewer
heads."""

import math

import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_topk_gb300 import workloads as W
from dsa_testlib import ensure_built, DeviceWorkload, OracleRows, check_sfa, check_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    return ensure_built()


def _oracle_idx(orc, wl):
    return np.stack([orc.topk(r)[0] for r in range(wl.n_q)]).astype(np.int32)


CASES = {
    "tiny": lambda: W.make("tiny"),
    "short_ctx": lambda: W.make("short_ctx"),
    "ragged_h100": lambda: W.custom([300, 1, 2500, 129], h_i=16, h_s=100, topk=256, seed=17),
    "mtp_h128": lambda: W.custom([1500, 700], per_seq=2, h_i=16, h_s=128, topk=512, seed=18),
    # 20 rows -> 7 splits per row, 40 rows -> 3: split counts that do not divide the 64
    # tiles of a 2048-entry row evenly
    "rows20_split7": lambda: W.custom([300 + 37 * i for i in range(20)], h_i=8, h_s=32, topk=256, seed=19),
    "rows40_split3": lambda: W.custom([200 + 11 * i for i in range(40)], h_i=8, h_s=48, topk=128, seed=20),
}


@pytest.mark.parametrize("name", list(CASES))
def test_sfa_matches_oracle(dsa, name):
    wl = CASES[name]()
    dw = DeviceWorkload(wl)
    orc = OracleRows(wl)
    idx = _oracle_idx(orc, wl)
    out, lse = dw.sparse_attn(torch.from_numpy(idx).cuda())
    assert dsa.device_status() == 0
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    qs = wl.q_sfa().double().numpy()
    for r in range(wl.n_q):
        o_ref, lse_ref = orc.sfa(r, idx[r], qs[r])
        check_sfa(out[r], o_ref)
        kvh = orc.kv_hat_rows(int(wl.q_seq[r]), idx[r])
        check_lse(lse[r], qs[r], kvh, idx[r], wl.sm_scale, lse_ref)


def test_sfa_padding_order_empty_and_bad_index(dsa):
    wl = W.custom([400, 90], h_i=8, h_s=32, topk=64, seed=19)
    dw = DeviceWorkload(wl)
    orc = OracleRows(wl)
    rng = np.random.default_rng(3)
    idx = np.full((2, 64), -1, np.int32)
    idx[0, 5:45] = rng.choice(400, 40, replace=False)      # padding on both sides
    out, lse = dw.sparse_attn(torch.from_numpy(idx).cuda())
    assert dsa.device_status() == 0
    qs = wl.q_sfa().double().numpy()
    o_ref, _ = orc.sfa(0, idx[0], qs[0])
    check_sfa(out[0].float().cpu().numpy(), o_ref)
    # row 1 is empty: zeros and -inf
    assert not out[1].float().abs().sum().item()
    assert torch.all(torch.isneginf(lse[1]))
    # reversing the index order changes nothing beyond rounding
    idx2 = idx.copy()
    idx2[0] = idx[0][::-1]
    out2, _ = dw.sparse_attn(torch.from_numpy(idx2).cuda())
    assert (out2[0].float() - out[0].float()).abs().max().item() <= 1e-2
    # an index past the sequence end is skipped and flagged
    idx3 = idx.copy()
    idx3[1, 0] = 90
    out3, _ = dw.sparse_attn(torch.from_numpy(idx3).cuda())
    assert dsa.device_status() & 8
    assert not out3[1].float().abs().sum().item()


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode_b32_ctx32k", "mixed_b128", "long_mtp_b4_ctx128k", "prefill_4k_over_64k"])
def test_sfa_full_size_sampled(dsa, name):
    wl = W.make(name)
    dw = DeviceWorkload(wl)
    orc = OracleRows(wl)
    gpu_idx, _ = dw.indexer_topk(with_scores=False)
    idx = gpu_idx.cpu().numpy().copy()
    rows = [0, wl.n_q - 1]
    for r in rows:                      # sampled rows get the oracle's own selection
        idx[r] = orc.topk(r)[0]
    out, lse = dw.sparse_attn(torch.from_numpy(idx).cuda())
    assert dsa.device_status() == 0
    out = out.float().cpu().numpy()
    qs = wl.q_sfa(rows).double().numpy()
    for i, r in enumerate(rows):
        o_ref, lse_ref = orc.sfa(r, idx[r], qs[i])
        check_sfa(out[r], o_ref)
        kvh = orc.kv_hat_rows(int(wl.q_seq[r]), idx[r])
        check_lse(lse.cpu().numpy()[r], qs[i], kvh, idx[r], wl.sm_scale, lse_ref)


def test_every_e4m3_code_dequantises_exactly(dsa):
    # One selected entry: its softmax weight is exactly 1, so the output row is the
    # dequantised V row itself.  The row's four 128-wide V tiles hold every non-NaN E4M3
    # code (positive codes, then negative ones), with the code 448 (0x7E) present so that
    # each tile's scale amax/448 is the power of two 2^e chosen below; every value
    # code * 2^e is exact in bf16, so the writer recovers the codes and the expected output
    # is exact.  Scales 2^-9 and 2^-100 push the subnormal codes' products far down.
    codes = np.arange(128)
    codes[0x7F] = 0x7E                      # 0x7F is NaN: use 448 again
    mag = oracle.codecs.e4m3_decode(codes)
    tiles = [mag, -mag, mag, -mag]          # codes 0x00..0x7E, then their negatives
    exps = [0, 5, -9, -100]
    v = np.concatenate([t * 2.0 ** e for t, e in zip(tiles, exps)] + [np.zeros(64)])
    wl = W.custom([64], h_i=8, h_s=16, topk=1, seed=3)
    kv = torch.zeros(64, 576, dtype=torch.float64)
    kv[5] = torch.from_numpy(v)
    kv = kv.to(torch.bfloat16)
    assert torch.equal(kv[5].double(), torch.from_numpy(v))  # exact in bf16
    kvc = dsa.alloc_kv_cache(wl.num_pages)
    dsa.quant_kv_fp8(kv.cuda(), torch.from_numpy(wl.slot_mapping(0)).cuda(), kvc)
    q = torch.randn(1, 16, 576, dtype=torch.float32).to(torch.bfloat16).cuda()
    idx = torch.tensor([[5]], dtype=torch.int32, device="cuda")
    out, _ = dsa.sparse_attn(q, kvc, torch.from_numpy(wl.page_table).cuda(),
                             torch.tensor([64], dtype=torch.int32, device="cuda"),
                             torch.zeros(1, dtype=torch.int32, device="cuda"), idx, wl.sm_scale)
    assert dsa.device_status() == 0
    got = out[0].double().cpu().numpy()
    want = np.broadcast_to(v[:512], got.shape)
    assert np.array_equal(got, want), np.argwhere(got != want)[:5]
