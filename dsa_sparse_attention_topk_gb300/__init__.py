"""GB300-native DeepSeek-style Sparse Attention decode path: thin Python binding.

Every call here only marshals arguments (device pointers, sizes, the current CUDA
stream) into the C ABI of ``libdsa.so`` (declared in ``include/dsa.h``); every step of
the path runs in the library's CUDA kernels.  If the library is missing or a call fails,
an exception is raised -- there is no other implementation to fall back to.

Functions (same names as the C entry points, without the ``dsa_`` prefix):

* ``quant_kv_mxfp8(k, slot_mapping, k_cache)``  -- cache writer, MXFP8 indexer keys
* ``quant_kv_fp8(kv, slot_mapping, kv_cache)``   -- cache writer, FP8 MLA latent rows
* ``quant_kv(k, kv, slot_mapping, k_cache, kv_cache)`` -- both writers in one launch
* ``decode_step(...)``  -- writers, indexer + Top-K and SFA of one decode step in one call
* ``indexer_topk(...)``                          -- fused Lightning Indexer + Top-K
* ``indexer_scores(...)``                        -- the same scores written in full
* ``sparse_attn(...)``                           -- Sparse Flash Attention
* ``device_status()``                            -- read and clear the device status word
"""

import ctypes
import os

import torch

from . import workloads  # noqa: F401  (seeded inputs; no computation of the method)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

PAGE_SIZE = 64
INDEX_DIM = 128
LATENT_DIM = 576
V_DIM = 512
KCACHE_PAGE_BYTES = 8448
KVCACHE_TOKEN_BYTES = 608

STATUS_BITS = {1: "BAD_PAGE", 2: "BAD_SEQ", 4: "BAD_LEN", 8: "BAD_INDEX", 16: "TIMEOUT", 32: "NAN_SCORE", 64: "INTERNAL"}

_lib = None


class DsaError(RuntimeError):
    """A non-zero return of the C ABI."""

    def __init__(self, code, msg):
        super().__init__(f"dsa error {code}: {msg}")
        self.code = code


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F32 = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGS = {
    "dsa_quant_kv_mxfp8": (ctypes.c_int, [_P, _P, _I32, _P, _I64, _P]),
    "dsa_quant_kv_fp8": (ctypes.c_int, [_P, _P, _I32, _P, _I64, _P]),
    "dsa_quant_kv": (ctypes.c_int, [_P, _P, _P, _I32, _P, _P, _I64, _P]),
    "dsa_indexer_topk": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _I64, _P, _I32, _P, _P, _P,
                                        _I32, _I32, _I32, _P, _P, _P]),
    "dsa_indexer_scores": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _I64, _P, _I32, _P, _P, _P,
                                          _I32, _I32, _P, _P]),
    "dsa_sparse_attn_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "dsa_sparse_attn": (ctypes.c_int, [_P, _I32, _I32, _P, _I64, _P, _I32, _P, _P, _I32, _P, _I32,
                                       _F32, _P, _P, _P, _SZ, _P]),
    "dsa_sparse_attn_noalloc": (ctypes.c_int, [_P, _I32, _I32, _P, _I64, _P, _I32, _P, _P, _I32, _P, _I32,
                                               _F32, _P, _P, _P]),
    "dsa_decode_step": (ctypes.c_int, [_P, _P, _P, _I32, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _I32,
                                       _P, _P, _I32, _P, _P, _I32, _I32, _P, _P, _I32, _F32, _P, _P, _P, _SZ,
                                       _P]),
    "dsa_device_status": (ctypes.c_int, [_P]),
    "dsa_test_stall_indexer": (ctypes.c_int, [_I32]),
    "dsa_topk_merge": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P]),
    "dsa_lse_combine": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _P, _P]),
    "dsa_last_error": (ctypes.c_char_p, []),
    "dsa_version": (ctypes.c_int, []),
}

SYMBOLS = tuple(_SIGS)


def lib():
    """Load libdsa.so once (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "or python -m dsa_sparse_attention_topk_gb300.build")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


def _check(rc):
    if rc != 0:
        raise DsaError(rc, lib().dsa_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, name):
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


# ---- cache allocation (plain torch allocations of the documented layouts) ----------

def alloc_k_cache(num_pages, device="cuda"):
    return torch.zeros(num_pages * KCACHE_PAGE_BYTES, dtype=torch.uint8, device=device)


def alloc_kv_cache(num_pages, device="cuda"):
    return torch.zeros(num_pages * PAGE_SIZE * KVCACHE_TOKEN_BYTES, dtype=torch.uint8, device=device)


# ---- entry points --------------------------------------------------------------------

def quant_kv_mxfp8(k, slot_mapping, k_cache, stream=None):
    """k: bf16 [n, 128]; slot_mapping: int64 [n]; k_cache: uint8 buffer of whole pages."""
    _need(k, torch.bfloat16, "k")
    _need(slot_mapping, torch.int64, "slot_mapping")
    num_slots = k_cache.numel() // KCACHE_PAGE_BYTES * PAGE_SIZE
    _check(lib().dsa_quant_kv_mxfp8(_ptr(k), _ptr(slot_mapping), k.shape[0], _ptr(k_cache),
                                    num_slots, _stream(stream)))


def quant_kv_fp8(kv, slot_mapping, kv_cache, stream=None):
    """kv: bf16 [n, 576]; slot_mapping: int64 [n]; kv_cache: uint8 buffer of whole pages."""
    _need(kv, torch.bfloat16, "kv")
    _need(slot_mapping, torch.int64, "slot_mapping")
    num_slots = kv_cache.numel() // (PAGE_SIZE * KVCACHE_TOKEN_BYTES) * PAGE_SIZE
    _check(lib().dsa_quant_kv_fp8(_ptr(kv), _ptr(slot_mapping), kv.shape[0], _ptr(kv_cache),
                                  num_slots, _stream(stream)))


def quant_kv(k, kv, slot_mapping, k_cache, kv_cache, stream=None):
    """Both cache writers in one launch: k bf16 [n, 128] -> k_cache, kv bf16 [n, 576] ->
    kv_cache, at the same int64 slots [n]."""
    _need(k, torch.bfloat16, "k")
    _need(kv, torch.bfloat16, "kv")
    _need(slot_mapping, torch.int64, "slot_mapping")
    if k.shape[0] != kv.shape[0] or k.shape[0] != slot_mapping.shape[0]:
        raise ValueError("quant_kv: k, kv and slot_mapping must have the same number of tokens")
    num_slots = min(k_cache.numel() // KCACHE_PAGE_BYTES,
                    kv_cache.numel() // (PAGE_SIZE * KVCACHE_TOKEN_BYTES)) * PAGE_SIZE
    _check(lib().dsa_quant_kv(_ptr(k), _ptr(kv), _ptr(slot_mapping), k.shape[0], _ptr(k_cache), _ptr(kv_cache),
                              num_slots, _stream(stream)))


def indexer_topk(q, w, k_cache, page_table, seq_lens, q_seq, q_pos, topk, max_ctx,
                 q_group=1, out_idx=None, out_scores=None, stream=None):
    """Fused indexer + Top-K.  q: bf16 [n_q, h_i, 128]; w: fp32 [n_q, h_i];
    page_table: int32 [n_seq, max_pages]; seq_lens: int32 [n_seq]; q_seq, q_pos: int32
    [n_q].  Returns (out_idx int32 [n_q, topk], out_scores fp32 or None)."""
    n_q, h_i, _ = q.shape
    if out_idx is None:
        out_idx = torch.empty(n_q, topk, dtype=torch.int32, device=q.device)
    num_pages = k_cache.numel() // KCACHE_PAGE_BYTES
    _check(lib().dsa_indexer_topk(_ptr(q), _ptr(w), n_q, h_i, q_group, _ptr(k_cache), num_pages,
                                  _ptr(page_table), page_table.shape[1], _ptr(seq_lens), _ptr(q_seq),
                                  _ptr(q_pos), seq_lens.shape[0], max_ctx, topk, _ptr(out_idx),
                                  _ptr(out_scores), _stream(stream)))
    return out_idx, out_scores


def indexer_scores(q, w, k_cache, page_table, seq_lens, q_seq, q_pos, max_ctx, q_group=1,
                   out=None, stream=None):
    """All scores [n_q, max_ctx] fp32 (-inf where a row may not select)."""
    n_q, h_i, _ = q.shape
    if out is None:
        out = torch.empty(n_q, max_ctx, dtype=torch.float32, device=q.device)
    num_pages = k_cache.numel() // KCACHE_PAGE_BYTES
    _check(lib().dsa_indexer_scores(_ptr(q), _ptr(w), n_q, h_i, q_group, _ptr(k_cache), num_pages,
                                    _ptr(page_table), page_table.shape[1], _ptr(seq_lens), _ptr(q_seq),
                                    _ptr(q_pos), seq_lens.shape[0], max_ctx, _ptr(out), _stream(stream)))
    return out


def sparse_attn_workspace_size(n_q, h_s, topk):
    return int(lib().dsa_sparse_attn_workspace_size(n_q, h_s, topk))


def sparse_attn(q, kv_cache, page_table, seq_lens, q_seq, topk_idx, sm_scale, out=None,
                out_lse=None, workspace=None, stream=None):
    """Sparse Flash Attention.  q: bf16 [n_q, h_s, 576]; topk_idx: int32 [n_q, K].
    Returns (out bf16 [n_q, h_s, 512], out_lse or None)."""
    n_q, h_s, _ = q.shape
    topk = topk_idx.shape[1]
    if out is None:
        out = torch.empty(n_q, h_s, V_DIM, dtype=torch.bfloat16, device=q.device)
    ws_need = sparse_attn_workspace_size(n_q, h_s, topk)
    if workspace is None and ws_need:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    num_pages = kv_cache.numel() // (PAGE_SIZE * KVCACHE_TOKEN_BYTES)
    _check(lib().dsa_sparse_attn(_ptr(q), n_q, h_s, _ptr(kv_cache), num_pages, _ptr(page_table),
                                 page_table.shape[1], _ptr(seq_lens), _ptr(q_seq), seq_lens.shape[0],
                                 _ptr(topk_idx), topk, float(sm_scale), _ptr(out), _ptr(out_lse),
                                 _ptr(workspace), 0 if workspace is None else workspace.numel(),
                                 _stream(stream)))
    return out, out_lse


def decode_step(k_new, kv_new, slot_mapping, k_cache, kv_cache, q_idx, w, q_sfa, page_table, seq_lens,
                q_seq, q_pos, topk, max_ctx, sm_scale, q_group=1, out_idx=None, out=None, out_lse=None,
                workspace=None, stream=None):
    """One decode step in one call: write k_new / kv_new (bf16 [n_new, 128] / [n_new, 576],
    int64 slots [n_new]) into the caches, then the fused indexer + Top-K, then Sparse Flash
    Attention over the selected entries.  Returns (out bf16 [n_q, h_s, 512], out_lse or
    None, out_idx int32 [n_q, topk])."""
    _need(k_new, torch.bfloat16, "k_new")
    _need(kv_new, torch.bfloat16, "kv_new")
    _need(slot_mapping, torch.int64, "slot_mapping")
    n_new = k_new.shape[0]
    if kv_new.shape[0] != n_new or slot_mapping.shape[0] != n_new:
        raise ValueError("decode_step: k_new, kv_new and slot_mapping must have the same number of tokens")
    n_q, h_i, _ = q_idx.shape
    h_s = q_sfa.shape[1]
    if out_idx is None:
        out_idx = torch.empty(n_q, topk, dtype=torch.int32, device=q_idx.device)
    if out is None:
        out = torch.empty(n_q, h_s, V_DIM, dtype=torch.bfloat16, device=q_idx.device)
    ws_need = sparse_attn_workspace_size(n_q, h_s, topk)
    if workspace is None and ws_need:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q_idx.device)
    num_pages = min(k_cache.numel() // KCACHE_PAGE_BYTES, kv_cache.numel() // (PAGE_SIZE * KVCACHE_TOKEN_BYTES))
    _check(lib().dsa_decode_step(_ptr(k_new), _ptr(kv_new), _ptr(slot_mapping), n_new, _ptr(k_cache),
                                 _ptr(kv_cache), num_pages, _ptr(page_table), page_table.shape[1],
                                 _ptr(seq_lens), seq_lens.shape[0], max_ctx, n_q, _ptr(q_seq), _ptr(q_pos),
                                 q_group, _ptr(q_idx), _ptr(w), h_i, topk, _ptr(out_idx), _ptr(q_sfa), h_s,
                                 float(sm_scale), _ptr(out), _ptr(out_lse), _ptr(workspace),
                                 0 if workspace is None else workspace.numel(), _stream(stream)))
    return out, out_lse, out_idx


def sparse_attn_noalloc(q, kv_cache, page_table, seq_lens, q_seq, topk_idx, sm_scale, out=None,
                        out_lse=None, stream=None):
    """Sparse Flash Attention with the split-merge scratch kept in the library's fixed
    array, for callers that cannot allocate device memory.  Same result as sparse_attn.
    Calls that overlap on the GPU share that array and must not run concurrently."""
    n_q, h_s, _ = q.shape
    topk = topk_idx.shape[1]
    if out is None:
        out = torch.empty(n_q, h_s, V_DIM, dtype=torch.bfloat16, device=q.device)
    num_pages = kv_cache.numel() // (PAGE_SIZE * KVCACHE_TOKEN_BYTES)
    _check(lib().dsa_sparse_attn_noalloc(_ptr(q), n_q, h_s, _ptr(kv_cache), num_pages, _ptr(page_table),
                                         page_table.shape[1], _ptr(seq_lens), _ptr(q_seq), seq_lens.shape[0],
                                         _ptr(topk_idx), topk, float(sm_scale), _ptr(out), _ptr(out_lse),
                                         _stream(stream)))
    return out, out_lse


NOALLOC_SCRATCH_BYTES = 40 * 1024 * 1024


def topk_merge(cand_idx, cand_scores, topk, part_offsets=None, local_lo=None, local_hi=None, out_idx=None,
               out_scores=None, stream=None):
    """The K highest of several parts' candidates per row (context parallelism).
    cand_idx int32 / cand_scores fp32 [n_parts, n_q, k_in] (part-local positions, -1 empty);
    part_offsets int32 [n_parts, n_q] or None.  Returns (out_idx int32 [n_q, topk] global
    positions by score then position, out_scores fp32, out_local int32 [n_q, topk] or None:
    the positions inside [local_lo, local_hi) relative to local_lo, -1 elsewhere)."""
    _need(cand_idx, torch.int32, "cand_idx")
    _need(cand_scores, torch.float32, "cand_scores")
    n_parts, n_q, k_in = cand_idx.shape
    if out_idx is None:
        out_idx = torch.empty(n_q, topk, dtype=torch.int32, device=cand_idx.device)
    if out_scores is None:
        out_scores = torch.empty(n_q, topk, dtype=torch.float32, device=cand_idx.device)
    out_local = None
    if local_lo is not None:
        out_local = torch.empty(n_q, topk, dtype=torch.int32, device=cand_idx.device)
    _check(lib().dsa_topk_merge(_ptr(cand_idx), _ptr(cand_scores), _ptr(part_offsets), n_parts, n_q, k_in, topk,
                                _ptr(out_idx), _ptr(out_scores), _ptr(local_lo), _ptr(local_hi), _ptr(out_local),
                                _stream(stream)))
    return out_idx, out_scores, out_local


def lse_combine(o_parts, lse_parts, out=None, out_lse=None, stream=None):
    """Combine attention outputs over disjoint entry sets: o_parts bf16 [n_parts, n_q, h, 512],
    lse_parts fp32 [n_parts, n_q, h].  Returns (out bf16 [n_q, h, 512], out_lse fp32)."""
    _need(o_parts, torch.bfloat16, "o_parts")
    _need(lse_parts, torch.float32, "lse_parts")
    n_parts, n_q, h, _ = o_parts.shape
    if out is None:
        out = torch.empty(n_q, h, V_DIM, dtype=torch.bfloat16, device=o_parts.device)
    if out_lse is None:
        out_lse = torch.empty(n_q, h, dtype=torch.float32, device=o_parts.device)
    _check(lib().dsa_lse_combine(_ptr(o_parts), _ptr(lse_parts), n_parts, n_q, h, _ptr(out), _ptr(out_lse),
                                 _stream(stream)))
    return out, out_lse


def device_status(stream=None):
    """Synchronise the stream and return (and clear) the device status bits."""
    rc = lib().dsa_device_status(_stream(stream))
    if rc < 0:
        _check(rc)
    return rc


def test_stall_indexer(wait_limit_us):
    """Testing aid for the bounded waits (dsa_test_stall_indexer): a positive limit makes
    every following indexer launch stall its copy producer and give up waiting after that
    many microseconds; 0 restores normal operation."""
    _check(lib().dsa_test_stall_indexer(int(wait_limit_us)))


def status_names(bits):
    return [n for b, n in STATUS_BITS.items() if bits & b]
