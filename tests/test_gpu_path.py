"""End-to-end GPU path (cache writers -> fused indexer + Top-K -> SFA) against the oracle,
and the invariances the method fixes: page placement does not matter, runs are
deterministic, a positive rescale of the head weights keeps the selection, and bad
inputs are reported through the device status word instead of faulting."""

import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_topk_gb300 import workloads as W
from dsa_testlib import ensure_built, DeviceWorkload, OracleRows, check_sfa, check_topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    return ensure_built()


def _end_to_end(dsa, wl, rows):
    dw = DeviceWorkload(wl)
    idx, vals = dw.indexer_topk()
    out, lse = dw.sparse_attn(idx)
    assert dsa.device_status() == 0
    idx = idx.cpu().numpy()
    out = out.float().cpu().numpy()
    orc = OracleRows(wl)
    qs = wl.q_sfa(rows).double().numpy()
    same = 0
    for i, r in enumerate(rows):
        ref_idx, s, mag = orc.topk(r)
        ndiff = check_topk(idx[r], vals[r].cpu().numpy(), s, mag, wl.topk)
        same += ndiff == 0
        # the attention over the GPU's own selection (equal to the oracle's up to
        # exchanges inside the tie band, which check_topk has just bounded)
        o_ref, _ = orc.sfa(r, idx[r], qs[i])
        check_sfa(out[r], o_ref)
    print(f"{wl.name}: {len(rows)} rows compared, {same} with the oracle's exact selection")


@pytest.mark.parametrize("name", ["tiny", "short_ctx"])
def test_end_to_end_small(dsa, name):
    wl = W.make(name)
    _end_to_end(dsa, wl, list(range(wl.n_q)))


@pytest.mark.slow
def test_end_to_end_bench_workload(dsa):
    wl = W.make("decode_b32_ctx32k")
    _end_to_end(dsa, wl, [0, 13, 31])


def test_page_placement_invariance(dsa):
    wl = W.custom([700, 300, 1500], h_i=16, h_s=32, topk=128, seed=23)
    a = DeviceWorkload(wl)
    b = DeviceWorkload(wl.identity_pages())
    ia, va = a.indexer_topk()
    ib, vb = b.indexer_topk()
    sa = np.sort(ia.cpu().numpy(), axis=1)
    sb = np.sort(ib.cpu().numpy(), axis=1)
    assert np.array_equal(sa, sb)
    oa, _ = a.sparse_attn(ia)
    ob, _ = b.sparse_attn(ia)
    assert torch.equal(oa, ob)


def test_determinism(dsa):
    wl = W.custom([2000, 333], h_i=64, h_s=64, topk=256, seed=24)
    dw = DeviceWorkload(wl)
    i1, v1 = dw.indexer_topk()
    i2, v2 = dw.indexer_topk()
    assert torch.equal(i1, i2) and torch.equal(v1, v2)
    o1, l1 = dw.sparse_attn(i1)
    o2, l2 = dw.sparse_attn(i1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_positive_weight_rescale_keeps_selection(dsa):
    wl = W.custom([3000], h_i=32, topk=300, seed=25)
    dw = DeviceWorkload(wl, with_kv=False)
    i1, _ = dw.indexer_topk()
    dw.w = dw.w * 4.0   # exact in fp32: every score scales by 4, order unchanged
    i2, _ = dw.indexer_topk()
    assert np.array_equal(np.sort(i1.cpu().numpy(), 1), np.sort(i2.cpu().numpy(), 1))


def test_bad_page_and_length_are_flagged(dsa):
    wl = W.custom([200], h_i=8, h_s=16, topk=64, seed=26)
    dw = DeviceWorkload(wl)
    pt = dw.page_table.clone()
    pt[0, 1] = wl.num_pages + 5          # out of the pool
    import dsa_sparse_attention_topk_gb300 as d
    d.indexer_topk(dw.q_idx, dw.w, dw.k_cache, pt, dw.seq_lens, dw.q_seq, dw.q_pos, 64, wl.max_ctx)
    assert d.device_status() & 1
    lens = dw.seq_lens.clone()
    lens[0] = wl.max_ctx + 1             # longer than max_ctx
    d.indexer_topk(dw.q_idx, dw.w, dw.k_cache, dw.page_table, lens, dw.q_seq, dw.q_pos, 64, wl.max_ctx)
    assert d.device_status() & 4
    qs = dw.q_seq.clone()
    qs[0] = 7                            # no such sequence
    d.indexer_topk(dw.q_idx, dw.w, dw.k_cache, dw.page_table, dw.seq_lens, qs, dw.q_pos, 64, wl.max_ctx)
    assert d.device_status() & 2
    assert d.device_status() == 0


@pytest.mark.slow
def test_repeated_calls_with_l2_flush_stay_clean(dsa):
    # Back-to-back launches with cold caches change the relative speed of the pipeline
    # stages; every bounded wait must still see its barrier phases in order (a timeout
    # would set the TIMEOUT status bit) and the results must not change.
    wl = W.make("decode_b32_ctx32k")
    dw = DeviceWorkload(wl)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    idx0, val0 = dw.indexer_topk()
    full0 = dw.indexer_scores()
    out0, _ = dw.sparse_attn(idx0)
    assert dsa.device_status() == 0
    for _ in range(15):
        flush.zero_()
        idx, val = dw.indexer_topk()
        flush.zero_()
        full = dw.indexer_scores()
        flush.zero_()
        out, _ = dw.sparse_attn(idx0)
        assert torch.equal(idx, idx0) and torch.equal(val, val0)
        assert torch.equal(full, full0) and torch.equal(out, out0)
    assert dsa.device_status() == 0


def _step_inputs(wl, dw):
    """The rows of the query tokens themselves (the step's new tokens) and their slots."""
    k_new, kv_new, s_new = [], [], []
    for b in range(wl.B):
        pos = wl.q_pos[wl.q_seq == b]
        if pos.size == 0:
            continue
        k_new.append(wl.k_seq(b, dw.q_idx_cpu, dw.w_cpu)[pos])
        kv_new.append(wl.kv_seq(b)[pos])
        s_new.append(torch.from_numpy(wl.slot_mapping(b)[pos]))
    return (torch.cat(k_new).cuda(), torch.cat(kv_new).cuda(), torch.cat(s_new).cuda())


@pytest.mark.parametrize("name", ["tiny", "mtp", "decode_b32_ctx32k"])
def test_decode_step_equals_the_three_calls(dsa, name):
    # dsa_decode_step writes the new tokens and decodes in one call; its indexer reads all
    # but the K-cache before the writer finishes.  The new tokens' cache slots are wiped
    # first, so a K-cache read that overtook the writer would change the selection.
    wl = (W.custom([1000, 3000, 2], per_seq=2, h_i=64, h_s=64, topk=512, seed=8) if name == "mtp"
          else W.make(name))
    dw = DeviceWorkload(wl)
    k_new, kv_new, s_new = _step_inputs(wl, dw)
    kc0, vc0 = dw.k_cache.clone(), dw.kv_cache.clone()
    for kc, vc in ((kc0, vc0),):
        pages = kc.view(-1, 8448)
        for s in s_new.tolist():
            pages[s // 64, (s % 64) * 128:(s % 64) * 128 + 128] = 0x7E    # codes -> +448
            pages[s // 64, 8192 + (s % 64) * 4:8192 + (s % 64) * 4 + 4] = 0xFE   # scales -> 2^127
            vc.view(-1, 608)[s] = 0x7E
    # the three calls on one copy of the wiped caches
    ka, va = kc0.clone(), vc0.clone()
    dsa.quant_kv(k_new, kv_new, s_new, ka, va)
    idx_a, _ = dsa.indexer_topk(dw.q_idx, dw.w, ka, dw.page_table, dw.seq_lens, dw.q_seq, dw.q_pos, wl.topk,
                                wl.max_ctx, q_group=wl.q_group)
    lse_a = torch.empty(wl.n_q, wl.h_s, dtype=torch.float32, device="cuda")
    out_a, _ = dsa.sparse_attn(dw.q_sfa, va, dw.page_table, dw.seq_lens, dw.q_seq, idx_a, wl.sm_scale,
                               out_lse=lse_a)
    # one decode step on another
    kb, vb = kc0.clone(), vc0.clone()
    lse_b = torch.empty(wl.n_q, wl.h_s, dtype=torch.float32, device="cuda")
    out_b, _, idx_b = dsa.decode_step(k_new, kv_new, s_new, kb, vb, dw.q_idx, dw.w, dw.q_sfa, dw.page_table,
                                      dw.seq_lens, dw.q_seq, dw.q_pos, wl.topk, wl.max_ctx, wl.sm_scale,
                                      q_group=wl.q_group, out_lse=lse_b)
    assert dsa.device_status() == 0
    assert torch.equal(ka, kb) and torch.equal(va, vb)
    assert torch.equal(ka, dw.k_cache) and torch.equal(va, dw.kv_cache)   # the wipe was undone
    assert torch.equal(idx_a, idx_b)
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)


@pytest.mark.parametrize("name", ["tiny", "decode_b32_ctx32k"])
def test_captured_step_replays_the_eager_step(dsa, name):
    # DsaDecodeLayer.capture_step records one decode step (with a host -> device copy of
    # staged inputs first and a device -> host copy of the output last) in a CUDA graph;
    # its replays give the eager step's results bit for bit
    from dsa_sparse_attention_topk_gb300.layer import DsaDecodeLayer
    wl = W.make(name)
    dw = DeviceWorkload(wl)
    k_new, kv_new, s_new = _step_inputs(wl, dw)
    layer = DsaDecodeLayer(wl.num_pages, wl.h_i, wl.h_s, wl.topk, wl.sm_scale, "cuda")
    layer.k_cache.copy_(dw.k_cache)
    layer.kv_cache.copy_(dw.kv_cache)
    inputs = dict(k_new=k_new, kv_new=kv_new, slots_new=s_new, q_idx=dw.q_idx, w=dw.w, q_sfa=dw.q_sfa,
                  page_table=dw.page_table, seq_lens=dw.seq_lens, q_seq=dw.q_seq, q_pos=dw.q_pos)
    order = ("k_new", "kv_new", "slots_new", "q_idx", "w", "q_sfa", "page_table", "seq_lens", "q_seq", "q_pos")
    out_e, lse_e, idx_e = [t.clone() for t in layer.step(*[inputs[k] for k in order], wl.max_ctx, wl.q_group)]
    host_q = dw.q_sfa.cpu().pin_memory()
    staged = torch.zeros_like(dw.q_sfa)
    result = torch.zeros(out_e.shape, dtype=out_e.dtype).pin_memory()
    replay = layer.capture_step(dict(inputs, q_sfa=staged), wl.max_ctx, wl.q_group, stage=(host_q, staged),
                                result=result)
    for _ in range(2):
        replay()
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    assert torch.equal(replay.idx, idx_e)
    assert torch.equal(replay.out, out_e) and torch.equal(replay.lse, lse_e)
    assert torch.equal(result, out_e.cpu())
