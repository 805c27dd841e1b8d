// C ABI entry points (include/dsa.h): argument checking, the device status word and
// the per-thread error message.  Every compute step runs in the kernels behind
// dsa_launch.h; nothing here touches tensor data on the host.

#include <atomic>
#include <cstdint>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "dsa_common.cuh"
#include "dsa_launch.h"

namespace {

__device__ unsigned g_status_word;

thread_local std::string t_last_error;

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device address of the status word, looked up once per device with that device current.
unsigned* status_ptr() {
  static std::mutex mu;
  static unsigned* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned*>(p);
  }
  return ptrs[dev];
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// dsa_test_stall_indexer: 0 = normal operation, else the waits' limit in microseconds with
// the indexer's copy producer stalled
std::atomic<int> g_stall_wait_us{0};

void apply_test_hooks(dsa::IndexerArgs& a) {
  const int us = g_stall_wait_us.load(std::memory_order_relaxed);
  if (us > 0) {
    a.wait_ns = static_cast<uint64_t>(us) * 1000ull;
    a.stall_producer = 1;
  }
}

}  // namespace

bool dsa::device_info(DevInfo* out, const char** err) {
  static std::mutex mu;
  static DevInfo cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    *err = "no current CUDA device";
    return false;
  }
  if (dev < 0 || dev >= 64) {
    *err = "device ordinal out of range (the library serves ordinals 0..63)";
    return false;
  }
  std::lock_guard<std::mutex> lock(mu);
  DevInfo& d = cache[dev];
  if (!d.n_sm) {
    DevInfo q;
    if (cudaDeviceGetAttribute(&q.n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&q.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        q.n_sm <= 0) {
      *err = "device attribute query failed";
      return false;
    }
    d = q;
  }
  *out = d;
  return true;
}

extern "C" {

int dsa_version(void) { return 101; }

const char* dsa_last_error(void) { return t_last_error.c_str(); }

int dsa_quant_kv_mxfp8(const void* k_bf16, const int64_t* slot_mapping, int32_t n_tokens,
                       uint8_t* k_cache, int64_t num_slots, void* stream) {
  if (n_tokens < 0) return fail(DSA_ERR_INVALID_ARG, "quant_kv_mxfp8: n_tokens < 0");
  if (n_tokens == 0) return DSA_OK;
  if (!k_bf16 || !slot_mapping || !k_cache) return fail(DSA_ERR_INVALID_ARG, "quant_kv_mxfp8: null pointer");
  if (!aligned(k_bf16, 16) || !aligned(k_cache, 16) || !aligned(slot_mapping, 8))
    return fail(DSA_ERR_INVALID_ARG, "quant_kv_mxfp8: k_bf16/k_cache must be 16-byte aligned");
  if (num_slots <= 0 || num_slots % DSA_PAGE_SIZE)
    return fail(DSA_ERR_INVALID_ARG, "quant_kv_mxfp8: num_slots must be a positive multiple of 64");
  unsigned* st = status_ptr();
  if (!st) return fail(DSA_ERR_CUDA, "quant_kv_mxfp8: no CUDA device");
  cudaError_t e = dsa::launch_quant_mxfp8(k_bf16, slot_mapping, n_tokens, k_cache, num_slots, st,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSA_OK : cuda_fail(e, "quant_kv_mxfp8 launch");
}

int dsa_quant_kv_fp8(const void* kv_bf16, const int64_t* slot_mapping, int32_t n_tokens,
                     uint8_t* kv_cache, int64_t num_slots, void* stream) {
  if (n_tokens < 0) return fail(DSA_ERR_INVALID_ARG, "quant_kv_fp8: n_tokens < 0");
  if (n_tokens == 0) return DSA_OK;
  if (!kv_bf16 || !slot_mapping || !kv_cache) return fail(DSA_ERR_INVALID_ARG, "quant_kv_fp8: null pointer");
  if (!aligned(kv_bf16, 16) || !aligned(kv_cache, 16) || !aligned(slot_mapping, 8))
    return fail(DSA_ERR_INVALID_ARG, "quant_kv_fp8: kv_bf16/kv_cache must be 16-byte aligned");
  if (num_slots <= 0 || num_slots % DSA_PAGE_SIZE)
    return fail(DSA_ERR_INVALID_ARG, "quant_kv_fp8: num_slots must be a positive multiple of 64");
  unsigned* st = status_ptr();
  if (!st) return fail(DSA_ERR_CUDA, "quant_kv_fp8: no CUDA device");
  cudaError_t e = dsa::launch_quant_fp8(kv_bf16, slot_mapping, n_tokens, kv_cache, num_slots, st,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSA_OK : cuda_fail(e, "quant_kv_fp8 launch");
}

int dsa_quant_kv(const void* k_bf16, const void* kv_bf16, const int64_t* slot_mapping, int32_t n_tokens,
                 uint8_t* k_cache, uint8_t* kv_cache, int64_t num_slots, void* stream) {
  if (n_tokens < 0) return fail(DSA_ERR_INVALID_ARG, "quant_kv: n_tokens < 0");
  if (n_tokens == 0) return DSA_OK;
  if (!k_bf16 || !kv_bf16 || !slot_mapping || !k_cache || !kv_cache)
    return fail(DSA_ERR_INVALID_ARG, "quant_kv: null pointer");
  if (!aligned(k_bf16, 16) || !aligned(kv_bf16, 16) || !aligned(k_cache, 16) || !aligned(kv_cache, 16) ||
      !aligned(slot_mapping, 8))
    return fail(DSA_ERR_INVALID_ARG, "quant_kv: rows and caches must be 16-byte aligned");
  if (num_slots <= 0 || num_slots % DSA_PAGE_SIZE)
    return fail(DSA_ERR_INVALID_ARG, "quant_kv: num_slots must be a positive multiple of 64");
  unsigned* st = status_ptr();
  if (!st) return fail(DSA_ERR_CUDA, "quant_kv: no CUDA device");
  cudaError_t e = dsa::launch_quant_both(k_bf16, kv_bf16, slot_mapping, n_tokens, k_cache, kv_cache, num_slots, st,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSA_OK : cuda_fail(e, "quant_kv launch");
}

static int check_indexer(const char* who, const void* q_bf16, const float* w, int32_t n_q, int32_t h_i,
                         int32_t q_group, const uint8_t* k_cache, int64_t num_pages,
                         const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                         const int32_t* q_seq, const int32_t* q_pos, int32_t n_seq, int32_t max_ctx) {
  if (n_q < 0 || n_seq < 0) return fail(DSA_ERR_INVALID_ARG, "%s: negative n_q or n_seq", who);
  if (h_i < 1 || h_i > 64) return fail(DSA_ERR_UNSUPPORTED, "%s: h_i must be 1..64 (got %d)", who, h_i);
  if (q_group < 1 || q_group > 4) return fail(DSA_ERR_UNSUPPORTED, "%s: q_group must be 1..4", who);
  if (q_group * h_i > 256) return fail(DSA_ERR_UNSUPPORTED, "%s: q_group * h_i must be <= 256", who);
  if (n_q % q_group) return fail(DSA_ERR_INVALID_ARG, "%s: n_q must be a multiple of q_group", who);
  if (max_ctx < 1 || max_ctx > 262144) return fail(DSA_ERR_UNSUPPORTED, "%s: max_ctx must be 1..262144", who);
  if (max_pages < (max_ctx + DSA_PAGE_SIZE - 1) / DSA_PAGE_SIZE)
    return fail(DSA_ERR_INVALID_ARG, "%s: max_pages < ceil(max_ctx / 64)", who);
  if (num_pages < 1) return fail(DSA_ERR_INVALID_ARG, "%s: num_pages must be >= 1", who);
  if (n_q == 0) return DSA_OK;
  if (!q_bf16 || !w || !k_cache || !page_table || !seq_lens || !q_seq || !q_pos)
    return fail(DSA_ERR_INVALID_ARG, "%s: null pointer", who);
  if (!aligned(q_bf16, 16) || !aligned(k_cache, 16) || !aligned(w, 4))
    return fail(DSA_ERR_INVALID_ARG, "%s: q_bf16 and k_cache must be 16-byte aligned", who);
  return DSA_OK;
}

int dsa_indexer_topk(const void* q_bf16, const float* w, int32_t n_q, int32_t h_i,
                     int32_t q_group, const uint8_t* k_cache, int64_t num_pages,
                     const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                     const int32_t* q_seq, const int32_t* q_pos, int32_t n_seq,
                     int32_t max_ctx, int32_t topk, int32_t* out_idx, float* out_scores,
                     void* stream) {
  int rc = check_indexer("indexer_topk", q_bf16, w, n_q, h_i, q_group, k_cache, num_pages, page_table,
                         max_pages, seq_lens, q_seq, q_pos, n_seq, max_ctx);
  if (rc) return rc;
  if (topk < 1 || topk > 2048) return fail(DSA_ERR_UNSUPPORTED, "indexer_topk: topk must be 1..2048");
  if (n_q == 0) return DSA_OK;
  if (!out_idx) return fail(DSA_ERR_INVALID_ARG, "indexer_topk: out_idx is null");
  unsigned* st = status_ptr();
  if (!st) return fail(DSA_ERR_CUDA, "indexer_topk: no CUDA device");
  dsa::IndexerArgs a{q_bf16, w, n_q, h_i, q_group, k_cache, num_pages, page_table, max_pages,
                     seq_lens, q_seq, q_pos, n_seq, max_ctx, topk, out_idx, out_scores, nullptr, st};
  apply_test_hooks(a);
  const char* why = nullptr;
  cudaError_t e = dsa::launch_indexer(a, static_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return why ? fail(DSA_ERR_UNSUPPORTED, "%s", why) : cuda_fail(e, "indexer_topk launch");
  return DSA_OK;
}

int dsa_indexer_scores(const void* q_bf16, const float* w, int32_t n_q, int32_t h_i,
                       int32_t q_group, const uint8_t* k_cache, int64_t num_pages,
                       const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                       const int32_t* q_seq, const int32_t* q_pos, int32_t n_seq,
                       int32_t max_ctx, float* out_scores, void* stream) {
  int rc = check_indexer("indexer_scores", q_bf16, w, n_q, h_i, q_group, k_cache, num_pages, page_table,
                         max_pages, seq_lens, q_seq, q_pos, n_seq, max_ctx);
  if (rc) return rc;
  if (n_q == 0) return DSA_OK;
  if (!out_scores) return fail(DSA_ERR_INVALID_ARG, "indexer_scores: out_scores is null");
  unsigned* st = status_ptr();
  if (!st) return fail(DSA_ERR_CUDA, "indexer_scores: no CUDA device");
  dsa::IndexerArgs a{q_bf16, w, n_q, h_i, q_group, k_cache, num_pages, page_table, max_pages,
                     seq_lens, q_seq, q_pos, n_seq, max_ctx, 1, nullptr, nullptr, out_scores, st};
  apply_test_hooks(a);
  const char* why = nullptr;
  cudaError_t e = dsa::launch_indexer(a, static_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return why ? fail(DSA_ERR_UNSUPPORTED, "%s", why) : cuda_fail(e, "indexer_scores launch");
  return DSA_OK;
}

size_t dsa_sparse_attn_workspace_size(int32_t n_q, int32_t h_s, int32_t topk) {
  if (n_q <= 0 || h_s <= 0 || topk <= 0) return 0;
  return dsa::sfa_workspace_bytes(n_q, h_s, topk);
}

int dsa_sparse_attn(const void* q_bf16, int32_t n_q, int32_t h_s, const uint8_t* kv_cache,
                    int64_t num_pages, const int32_t* page_table, int32_t max_pages,
                    const int32_t* seq_lens, const int32_t* q_seq, int32_t n_seq,
                    const int32_t* topk_idx, int32_t topk, float sm_scale, void* out_bf16,
                    float* out_lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (n_q < 0 || n_seq < 0) return fail(DSA_ERR_INVALID_ARG, "sparse_attn: negative n_q or n_seq");
  if (h_s < 1 || h_s > 128) return fail(DSA_ERR_UNSUPPORTED, "sparse_attn: h_s must be 1..128");
  if (topk < 1 || topk > 65536) return fail(DSA_ERR_UNSUPPORTED, "sparse_attn: topk must be 1..65536");
  if (max_pages < 1 || num_pages < 1) return fail(DSA_ERR_INVALID_ARG, "sparse_attn: max_pages and num_pages must be >= 1");
  if (!(sm_scale > 0.f) || sm_scale != sm_scale) return fail(DSA_ERR_INVALID_ARG, "sparse_attn: sm_scale must be positive");
  if (n_q == 0) return DSA_OK;
  if (!q_bf16 || !kv_cache || !page_table || !seq_lens || !q_seq || !topk_idx || !out_bf16)
    return fail(DSA_ERR_INVALID_ARG, "sparse_attn: null pointer");
  if (!aligned(q_bf16, 16) || !aligned(kv_cache, 16) || !aligned(out_bf16, 16))
    return fail(DSA_ERR_INVALID_ARG, "sparse_attn: q, kv_cache and out must be 16-byte aligned");
  const size_t need = dsa::sfa_workspace_bytes(n_q, h_s, topk);
  if (need && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
    return fail(DSA_ERR_INVALID_ARG, "sparse_attn: workspace must be >= %zu bytes and 256-byte aligned", need);
  unsigned* st = status_ptr();
  if (!st) return fail(DSA_ERR_CUDA, "sparse_attn: no CUDA device");
  dsa::SfaArgs a{q_bf16, n_q, h_s, kv_cache, num_pages, page_table, max_pages, seq_lens, q_seq, n_seq,
                 topk_idx, topk, sm_scale, out_bf16, out_lse, workspace, workspace_bytes, st};
  const char* why = nullptr;
  cudaError_t e = dsa::launch_sfa(a, static_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return why ? fail(DSA_ERR_UNSUPPORTED, "%s", why) : cuda_fail(e, "sparse_attn launch");
  return DSA_OK;
}

int dsa_decode_step(const void* k_new_bf16, const void* kv_new_bf16, const int64_t* slot_mapping, int32_t n_new,
                    uint8_t* k_cache, uint8_t* kv_cache, int64_t num_pages, const int32_t* page_table,
                    int32_t max_pages, const int32_t* seq_lens, int32_t n_seq, int32_t max_ctx, int32_t n_q,
                    const int32_t* q_seq, const int32_t* q_pos, int32_t q_group, const void* q_idx_bf16,
                    const float* w, int32_t h_i, int32_t topk, int32_t* out_idx, const void* q_sfa_bf16,
                    int32_t h_s, float sm_scale, void* out_bf16, float* out_lse, void* workspace,
                    size_t workspace_bytes, void* stream) {
  // every argument is checked before anything is launched
  if (n_new < 0) return fail(DSA_ERR_INVALID_ARG, "decode_step: n_new < 0");
  if (num_pages < 1 || num_pages > INT64_MAX / DSA_PAGE_SIZE)
    return fail(DSA_ERR_INVALID_ARG, "decode_step: num_pages must be >= 1");
  if (n_new > 0) {
    if (!k_new_bf16 || !kv_new_bf16 || !slot_mapping || !k_cache || !kv_cache)
      return fail(DSA_ERR_INVALID_ARG, "decode_step: null pointer among the new tokens or caches");
    if (!aligned(k_new_bf16, 16) || !aligned(kv_new_bf16, 16) || !aligned(k_cache, 16) || !aligned(kv_cache, 16) ||
        !aligned(slot_mapping, 8))
      return fail(DSA_ERR_INVALID_ARG, "decode_step: rows and caches must be 16-byte aligned");
  }
  int rc = check_indexer("decode_step", q_idx_bf16, w, n_q, h_i, q_group, k_cache, num_pages, page_table,
                         max_pages, seq_lens, q_seq, q_pos, n_seq, max_ctx);
  if (rc) return rc;
  if (topk < 1 || topk > 2048) return fail(DSA_ERR_UNSUPPORTED, "decode_step: topk must be 1..2048");
  if (h_s < 1 || h_s > 128) return fail(DSA_ERR_UNSUPPORTED, "decode_step: h_s must be 1..128");
  if (!(sm_scale > 0.f) || sm_scale != sm_scale) return fail(DSA_ERR_INVALID_ARG, "decode_step: sm_scale must be positive");
  if (n_q > 0) {
    if (!out_idx || !q_sfa_bf16 || !kv_cache || !out_bf16) return fail(DSA_ERR_INVALID_ARG, "decode_step: null pointer");
    if (!aligned(q_sfa_bf16, 16) || !aligned(kv_cache, 16) || !aligned(out_bf16, 16))
      return fail(DSA_ERR_INVALID_ARG, "decode_step: q_sfa, kv_cache and out must be 16-byte aligned");
    const size_t need = dsa::sfa_workspace_bytes(n_q, h_s, topk);
    if (need && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
      return fail(DSA_ERR_INVALID_ARG, "decode_step: workspace must be >= %zu bytes and 256-byte aligned", need);
  }
  if (n_new == 0 && n_q == 0) return DSA_OK;  // nothing to launch
  unsigned* st = status_ptr();
  if (!st) return fail(DSA_ERR_CUDA, "decode_step: no CUDA device");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // one new token per query row (token i is row i's own token): the indexer writes them
  // itself, each before it loads the page that holds it; otherwise a writer launch first
  const bool fuse = n_new > 0 && n_new == n_q;
  cudaError_t e = cudaSuccess;
  if (!fuse) {
    e = dsa::launch_quant_both(k_new_bf16, kv_new_bf16, slot_mapping, n_new, k_cache, kv_cache,
                               num_pages * DSA_PAGE_SIZE, st, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode_step: cache writer launch");
  }
  if (n_q == 0) return DSA_OK;
  dsa::IndexerArgs ia{q_idx_bf16, w, n_q, h_i, q_group, k_cache, num_pages, page_table, max_pages,
                      seq_lens, q_seq, q_pos, n_seq, max_ctx, topk, out_idx, nullptr, nullptr, st};
  if (fuse) {
    ia.fuse_writes = 1;
    ia.k_new = k_new_bf16;
    ia.kv_new = kv_new_bf16;
    ia.slot_mapping = slot_mapping;
    ia.kv_cache = kv_cache;
    ia.num_slots = num_pages * DSA_PAGE_SIZE;
  } else {
    ia.early_inputs = n_new > 0 ? 1 : 0;  // the writer launched just above precedes the indexer
  }
  apply_test_hooks(ia);
  const char* why = nullptr;
  e = dsa::launch_indexer(ia, s, &why);
  if (e != cudaSuccess) return why ? fail(DSA_ERR_UNSUPPORTED, "%s", why) : cuda_fail(e, "decode_step: indexer launch");
  dsa::SfaArgs sa{q_sfa_bf16, n_q, h_s, kv_cache, num_pages, page_table, max_pages, seq_lens, q_seq, n_seq,
                  out_idx, topk, sm_scale, out_bf16, out_lse, workspace, workspace_bytes, st};
  e = dsa::launch_sfa(sa, s, &why);
  if (e != cudaSuccess) return why ? fail(DSA_ERR_UNSUPPORTED, "%s", why) : cuda_fail(e, "decode_step: sparse_attn launch");
  return DSA_OK;
}

int dsa_sparse_attn_noalloc(const void* q_bf16, int32_t n_q, int32_t h_s, const uint8_t* kv_cache,
                            int64_t num_pages, const int32_t* page_table, int32_t max_pages,
                            const int32_t* seq_lens, const int32_t* q_seq, int32_t n_seq,
                            const int32_t* topk_idx, int32_t topk, float sm_scale, void* out_bf16,
                            float* out_lse, void* stream) {
  if (n_q < 0 || n_seq < 0) return fail(DSA_ERR_INVALID_ARG, "sparse_attn_noalloc: negative n_q or n_seq");
  if (h_s < 1 || h_s > 128) return fail(DSA_ERR_UNSUPPORTED, "sparse_attn_noalloc: h_s must be 1..128");
  if (topk < 1 || topk > 65536) return fail(DSA_ERR_UNSUPPORTED, "sparse_attn_noalloc: topk must be 1..65536");
  if (max_pages < 1 || num_pages < 1)
    return fail(DSA_ERR_INVALID_ARG, "sparse_attn_noalloc: max_pages and num_pages must be >= 1");
  if (!(sm_scale > 0.f) || sm_scale != sm_scale)
    return fail(DSA_ERR_INVALID_ARG, "sparse_attn_noalloc: sm_scale must be positive");
  if (n_q == 0) return DSA_OK;
  if (!q_bf16 || !kv_cache || !page_table || !seq_lens || !q_seq || !topk_idx || !out_bf16)
    return fail(DSA_ERR_INVALID_ARG, "sparse_attn_noalloc: null pointer");
  if (!aligned(q_bf16, 16) || !aligned(kv_cache, 16) || !aligned(out_bf16, 16))
    return fail(DSA_ERR_INVALID_ARG, "sparse_attn_noalloc: q, kv_cache and out must be 16-byte aligned");
  const size_t need = dsa::sfa_workspace_bytes(n_q, h_s, topk);
  if (need > static_cast<size_t>(DSA_NOALLOC_SCRATCH_BYTES))
    return fail(DSA_ERR_UNSUPPORTED,
                "sparse_attn_noalloc: n_q=%d, h_s=%d, topk=%d need %zu bytes of scratch, more than the "
                "fixed %zu (use dsa_sparse_attn with a caller-allocated workspace)",
                n_q, h_s, topk, need, static_cast<size_t>(DSA_NOALLOC_SCRATCH_BYTES));
  unsigned* st = status_ptr();
  if (!st) return fail(DSA_ERR_CUDA, "sparse_attn_noalloc: no CUDA device");
  dsa::SfaArgs a{q_bf16, n_q, h_s, kv_cache, num_pages, page_table, max_pages, seq_lens, q_seq, n_seq,
                 topk_idx, topk, sm_scale, out_bf16, out_lse, nullptr, 0, st};
  const char* why = nullptr;
  cudaError_t e = dsa::launch_sfa_noalloc(a, static_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess)
    return why ? fail(DSA_ERR_UNSUPPORTED, "%s", why) : cuda_fail(e, "sparse_attn_noalloc launch");
  return DSA_OK;
}

int dsa_topk_merge(const int32_t* cand_idx, const float* cand_scores, const int32_t* part_offsets, int32_t n_parts,
                   int32_t n_q, int32_t k_in, int32_t topk, int32_t* out_idx, float* out_scores,
                   const int32_t* local_lo, const int32_t* local_hi, int32_t* out_local, void* stream) {
  if (n_q < 0) return fail(DSA_ERR_INVALID_ARG, "topk_merge: n_q < 0");
  if (n_parts < 1 || k_in < 1 || topk < 1) return fail(DSA_ERR_INVALID_ARG, "topk_merge: n_parts, k_in and topk must be >= 1");
  if (static_cast<int64_t>(n_parts) * k_in > 16384)
    return fail(DSA_ERR_UNSUPPORTED, "topk_merge: n_parts * k_in must be <= 16384 (got %lld)",
                static_cast<long long>(n_parts) * k_in);
  if (n_q == 0) return DSA_OK;
  if (!cand_idx || !cand_scores || !out_idx) return fail(DSA_ERR_INVALID_ARG, "topk_merge: null pointer");
  if ((out_local != nullptr) != (local_lo != nullptr && local_hi != nullptr))
    return fail(DSA_ERR_INVALID_ARG, "topk_merge: out_local needs local_lo and local_hi (and they need it)");
  unsigned* st = status_ptr();
  if (!st) return fail(DSA_ERR_CUDA, "topk_merge: no CUDA device");
  dsa::TopkMergeArgs a{cand_idx, cand_scores, part_offsets, n_parts, n_q, k_in, topk, out_idx, out_scores,
                       local_lo, local_hi, out_local, st};
  cudaError_t e = dsa::launch_topk_merge(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSA_OK : cuda_fail(e, "topk_merge launch");
}

int dsa_lse_combine(const void* o_parts, const float* lse_parts, int32_t n_parts, int32_t n_q, int32_t h,
                    void* out_bf16, float* out_lse, void* stream) {
  if (n_q < 0) return fail(DSA_ERR_INVALID_ARG, "lse_combine: n_q < 0");
  if (n_parts < 1 || h < 1 || h > 65535) return fail(DSA_ERR_INVALID_ARG, "lse_combine: n_parts >= 1 and h in 1..65535");
  if (n_q == 0) return DSA_OK;
  if (!o_parts || !lse_parts || !out_bf16) return fail(DSA_ERR_INVALID_ARG, "lse_combine: null pointer");
  if (!aligned(o_parts, 8) || !aligned(out_bf16, 8))
    return fail(DSA_ERR_INVALID_ARG, "lse_combine: o_parts and out must be 8-byte aligned");
  cudaError_t e = dsa::launch_lse_combine(o_parts, lse_parts, n_parts, n_q, h, out_bf16, out_lse,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSA_OK : cuda_fail(e, "lse_combine launch");
}

int dsa_test_stall_indexer(int32_t wait_limit_us) {
  if (wait_limit_us < 0 || wait_limit_us > 10000000)
    return fail(DSA_ERR_INVALID_ARG, "test_stall_indexer: wait_limit_us must be 0..10000000");
  g_stall_wait_us.store(wait_limit_us, std::memory_order_relaxed);
  return DSA_OK;
}

int dsa_device_status(void* stream) {
  unsigned* st = status_ptr();
  if (!st) return fail(DSA_ERR_CUDA, "device_status: no CUDA device");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, st, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(st, 0, sizeof(unsigned), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "device_status");
  return static_cast<int>(v);
}

}  // extern "C"
