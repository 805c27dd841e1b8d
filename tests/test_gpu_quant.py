"""GPU parity of the cache writers: codes and scales must be bit-exact with the oracle's
MXFP8 (group 32, OCP scale rule) and FP8 (per-128 tile, fp32 amax/448) quantisers."""

import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_topk_gb300 import workloads as W
from dsa_testlib import ensure_built, DeviceWorkload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    return ensure_built()


def _kcache_rows(cache, wl, b):
    pages = cache.cpu().numpy().reshape(-1, 8448)
    L = int(wl.seq_lens[b])
    p = np.arange(L)
    pg = wl.page_table[b, p // 64]
    r = p % 64
    codes = pages[pg[:, None], (r * 128)[:, None] + np.arange(128)[None, :]]
    scales = pages[pg[:, None], (8192 + r * 4)[:, None] + np.arange(4)[None, :]]
    return codes, scales


def _kvcache_rows(cache, slots):
    recs = cache.cpu().numpy().reshape(-1, 608)[slots]
    codes = recs[:, :576]
    scales = recs[:, 576:596].copy().view(np.float32)
    pad = recs[:, 596:608]
    return codes, scales, pad


@pytest.mark.parametrize("name,lens", [("tiny", None), ("ragged", [130, 1, 700, 64, 65])])
def test_cache_writers_bit_exact(dsa, name, lens):
    wl = W.make(name) if lens is None else W.custom(lens, h_i=8, outliers=4, seed=21)
    dw = DeviceWorkload(wl)
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    for b in range(wl.B):
        k = wl.k_seq(b).double().numpy()
        c_ref, s_ref = oracle.mxfp8_quantize(k)
        c, s = _kcache_rows(dw.k_cache, wl, b)
        assert np.array_equal(c, c_ref), f"seq {b}: {np.sum(c != c_ref)} MXFP8 codes differ"
        assert np.array_equal(s, s_ref), f"seq {b}: MXFP8 scales differ"
        kv = wl.kv_seq(b).double().numpy()
        vc_ref, vs_ref = oracle.fp8_tile_quantize(kv)
        vc, vs, pad = _kvcache_rows(dw.kv_cache, wl.slot_mapping(b))
        assert np.array_equal(vc, vc_ref), f"seq {b}: {np.sum(vc != vc_ref)} FP8 codes differ"
        assert np.array_equal(vs.view(np.uint32), vs_ref.view(np.uint32)), f"seq {b}: FP8 scales differ"
        assert not pad.any()


def _special_rows(width, n=64, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, width)).astype(np.float32)
    x[0] = 0.0
    x[1] = -0.0
    x[2] *= 1e-38          # bf16 subnormals
    x[3] *= 1e37
    x[4, ::3] = 0.0
    x[5] = np.where(np.arange(width) % 2 == 0, 448.0, -449.0)
    x[6] *= 2.0 ** -130
    x[7, :32] = -0.0
    x[8] = rng.integers(-3, 4, width)
    x[9] = np.float32(3.3895e38) * np.sign(x[9])   # close to the bf16 maximum
    return torch.from_numpy(x).to(torch.bfloat16)


def test_cache_writers_special_values_bit_exact(dsa):
    n = 64
    slots = torch.arange(n, dtype=torch.int64)
    k = _special_rows(128, n, 1)
    kv = _special_rows(576, n, 2)
    kc = dsa.alloc_k_cache(1)
    vc = dsa.alloc_kv_cache(1)
    dsa.quant_kv_mxfp8(k.cuda(), slots.cuda(), kc)
    dsa.quant_kv_fp8(kv.cuda(), slots.cuda(), vc)
    assert dsa.device_status() == 0
    page = kc.cpu().numpy()
    c_ref, s_ref = oracle.mxfp8_quantize(k.double().numpy())
    assert np.array_equal(page[:8192].reshape(64, 128), c_ref)
    assert np.array_equal(page[8192:].reshape(64, 4), s_ref)
    vc_ref, vs_ref = oracle.fp8_tile_quantize(kv.double().numpy())
    codes, scales, pad = _kvcache_rows(vc, np.arange(n))
    assert np.array_equal(codes, vc_ref)
    assert np.array_equal(scales.view(np.uint32), vs_ref.view(np.uint32))


def test_negative_slots_skip_and_out_of_range_slots_flag(dsa):
    k = _special_rows(128, 64, 3)[:4].contiguous().cuda()
    kc = dsa.alloc_k_cache(1)
    kc.fill_(0xAB)
    dsa.quant_kv_mxfp8(k, torch.tensor([-1, 0, 64, -5], dtype=torch.int64, device="cuda"), kc)
    bits = dsa.device_status()
    assert bits & 1, "slot 64 of a one-page cache must flag BAD_PAGE"
    page = kc.cpu().numpy()
    c_ref, _ = oracle.mxfp8_quantize(k.cpu().double().numpy())
    assert np.array_equal(page[:128], c_ref[1])      # token 1 -> slot 0
    assert np.all(page[128:8192] == 0xAB)             # nothing else written
    assert dsa.device_status() == 0                   # cleared by the read


def test_paired_writer_matches_the_oracle_and_skips_like_the_single_writers(dsa):
    # dsa_quant_kv writes both caches in one launch: the same codes and scales as the two
    # writers, checked against the oracle, with a skipped (-1) and an out-of-range slot
    n = 64
    k = _special_rows(128, n, 4)
    kv = _special_rows(576, n, 5)
    slots = torch.arange(n, dtype=torch.int64)
    slots[7] = -1
    slots[9] = 64  # past a one-page cache: skipped and flagged
    kc = dsa.alloc_k_cache(1)
    vc = dsa.alloc_kv_cache(1)
    kc.fill_(0xAB)
    vc.fill_(0xAB)
    dsa.quant_kv(k.cuda(), kv.cuda(), slots.cuda(), kc, vc)
    assert dsa.device_status() & 1, "slot 64 of a one-page cache must flag BAD_PAGE"
    written = np.array([i for i in range(n) if i not in (7, 9)])
    page = kc.cpu().numpy()
    c_ref, s_ref = oracle.mxfp8_quantize(k.double().numpy())
    assert np.array_equal(page[:8192].reshape(64, 128)[written], c_ref[written])
    assert np.array_equal(page[8192:].reshape(64, 4)[written], s_ref[written])
    assert np.all(page[:8192].reshape(64, 128)[[7, 9]] == 0xAB)
    vc_ref, vs_ref = oracle.fp8_tile_quantize(kv.double().numpy())
    codes, scales, _ = _kvcache_rows(vc, written)
    assert np.array_equal(codes, vc_ref[written])
    assert np.array_equal(scales.view(np.uint32), vs_ref[written].view(np.uint32))
    untouched, _, _ = _kvcache_rows(vc, np.array([7, 9]))
    assert np.all(untouched == 0xAB)
    assert dsa.device_status() == 0
