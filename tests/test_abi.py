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
    assert dsa.lib().dsa_version() == 100


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
