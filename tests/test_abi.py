"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every entry
point that include/dsa.h declares, and rejects bad arguments before launching anything."""

import ctypes
import os
import re

import pytest

from dsa_testlib import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dsa():
    return ensure_built()


def _declared():
    src = open(os.path.join(ROOT, "include", "dsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_path(dsa):
    names = _declared()
    for n in ["dsa_quant_kv_mxfp8", "dsa_quant_kv_fp8", "dsa_indexer_topk", "dsa_sparse_attn",
              "dsa_device_status", "dsa_last_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(dsa):
    h = ctypes.CDLL(dsa.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(h, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol(dsa):
    assert set(_declared()) == set(dsa.SYMBOLS)


def test_version(dsa):
    assert dsa.lib().dsa_version() == 101


def _idx_call(lib, **kw):
    a = dict(q=1, w=1, n_q=1, h_i=64, q_group=1, k_cache=16, num_pages=1, pt=1, max_pages=1,
             seq_lens=1, q_seq=1, q_pos=1, n_seq=1, max_ctx=64, topk=16, out_idx=4, out_scores=None)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.dsa_indexer_topk(P(a["q"] * 16), P(a["w"] * 16), a["n_q"], a["h_i"], a["q_group"],
                                P(a["k_cache"] * 16), a["num_pages"], P(a["pt"] * 16), a["max_pages"],
                                P(a["seq_lens"] * 16), P(a["q_seq"] * 16), P(a["q_pos"] * 16), a["n_seq"],
                                a["max_ctx"], a["topk"], P(a["out_idx"] * 16), a["out_scores"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(h_i=65), -2), (dict(h_i=0), -2), (dict(q_group=5), -2), (dict(q_group=4, h_i=65), -2),
    (dict(n_q=3, q_group=2), -1), (dict(topk=0), -2), (dict(topk=4096), -2),
    (dict(max_ctx=0), -2), (dict(max_ctx=300000), -2), (dict(max_ctx=129, max_pages=2), -1),
    (dict(q=0), -1), (dict(out_idx=0), -1), (dict(n_q=-1), -1), (dict(num_pages=0), -1),
])
def test_indexer_rejects_bad_arguments(dsa, kw, code):
    lib = dsa.lib()
    assert _idx_call(lib, **kw) == code
    assert lib.dsa_last_error()


def test_indexer_rejects_misaligned_pointers(dsa):
    lib = dsa.lib()
    P = ctypes.c_void_p
    rc = lib.dsa_indexer_topk(P(17), P(16), 1, 64, 1, P(32), 1, P(16), 1, P(16), P(16), P(16), 1, 64, 16,
                              P(64), None, None)
    assert rc == -1 and b"aligned" in lib.dsa_last_error()


def test_zero_rows_is_a_no_op(dsa):
    assert _idx_call(dsa.lib(), n_q=0, q=0, out_idx=0) == 0


def test_quant_and_sfa_reject_bad_arguments(dsa):
    lib = dsa.lib()
    P = ctypes.c_void_p
    assert lib.dsa_quant_kv_mxfp8(P(16), P(16), 4, P(16), 100, None) == -1     # not a page multiple
    assert lib.dsa_quant_kv_fp8(None, P(16), 4, P(16), 64, None) == -1
    assert lib.dsa_quant_kv_fp8(P(8), P(16), 4, P(16), 64, None) == -1        # misaligned source
    assert lib.dsa_quant_kv_mxfp8(P(16), P(16), 0, P(16), 64, None) == 0      # nothing to do
    assert lib.dsa_quant_kv(P(16), P(16), P(16), 4, P(16), P(16), 100, None) == -1   # not a page multiple
    assert lib.dsa_quant_kv(P(16), None, P(16), 4, P(16), P(16), 64, None) == -1     # no latent rows
    assert lib.dsa_quant_kv(P(16), P(16), P(16), 4, P(16), P(24), 64, None) == -1    # misaligned cache
    assert lib.dsa_quant_kv(P(16), P(16), P(16), -1, P(16), P(16), 64, None) == -1
    assert lib.dsa_quant_kv(None, None, None, 0, None, None, 64, None) == 0          # nothing to do
    args = [P(16), 1, 128, P(16), 1, P(16), 1, P(16), P(16), 1, P(16), 2048, ctypes.c_float(0.07),
            P(16), None, None, 0, None]
    bad_h = list(args); bad_h[2] = 129
    assert lib.dsa_sparse_attn(*bad_h) == -2
    bad_scale = list(args); bad_scale[12] = ctypes.c_float(0.0)
    assert lib.dsa_sparse_attn(*bad_scale) == -1
    bad_ptr = list(args); bad_ptr[13] = None
    assert lib.dsa_sparse_attn(*bad_ptr) == -1


def test_workspace_size_is_host_only(dsa):
    n = dsa.lib().dsa_sparse_attn_workspace_size(32, 128, 2048)
    assert n >= 0
    assert dsa.lib().dsa_sparse_attn_workspace_size(0, 128, 2048) == 0


def _step_call(lib, **kw):
    P = ctypes.c_void_p
    a = dict(k_new=1, kv_new=1, slots=1, n_new=2, k_cache=1, kv_cache=1, num_pages=4, pt=1, max_pages=4,
             seq_lens=1, n_seq=1, max_ctx=256, n_q=1, q_seq=1, q_pos=1, q_group=1, q_idx=1, w=1, h_i=64,
             topk=16, out_idx=1, q_sfa=1, h_s=128, sm_scale=0.07, out=1, lse=None, ws=1, ws_bytes=1 << 30)
    a.update(kw)
    p = lambda v: None if v is None else P(v * 256)
    return lib.dsa_decode_step(p(a["k_new"]), p(a["kv_new"]), p(a["slots"]), a["n_new"], p(a["k_cache"]),
                               p(a["kv_cache"]), a["num_pages"], p(a["pt"]), a["max_pages"], p(a["seq_lens"]),
                               a["n_seq"], a["max_ctx"], a["n_q"], p(a["q_seq"]), p(a["q_pos"]), a["q_group"],
                               p(a["q_idx"]), p(a["w"]), a["h_i"], a["topk"], p(a["out_idx"]), p(a["q_sfa"]),
                               a["h_s"], ctypes.c_float(a["sm_scale"]), p(a["out"]), p(a["lse"]), p(a["ws"]),
                               a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(n_new=-1), -1), (dict(kv_new=None), -1), (dict(num_pages=0), -1), (dict(h_i=65), -2),
    (dict(topk=4096), -2), (dict(h_s=129), -2), (dict(sm_scale=0.0), -1), (dict(out=None), -1),
    (dict(q_sfa=None), -1), (dict(ws=None, topk=2048), -1), (dict(n_q=3, q_group=2), -1),
])
def test_decode_step_rejects_bad_arguments_before_launching(dsa, kw, code):
    lib = dsa.lib()
    assert _step_call(lib, **kw) == code
    assert lib.dsa_last_error()


def test_decode_step_with_nothing_to_do(dsa):
    # no new tokens and no query rows: nothing to launch
    assert _step_call(dsa.lib(), n_new=0, n_q=0, k_new=None, kv_new=None, slots=None) == 0
