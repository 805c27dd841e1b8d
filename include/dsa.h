/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DeepSeek-style Sparse Attention decode path.
 *
 * The path has two stages, as described on "Deep Dive into Sparse Attention and
 * Engineering Optimizations for Efficient Inference in Kimi K3.1 Pro" (section 1: a cheap
 * pass picks the positions, then exact attention runs only on those):
 *   1. a fused Lightning Indexer that reads an MXFP8 K-cache straight from its pages,
 *      scores every selectable past position and keeps the Top-K on chip
 *      (dsa_indexer_topk);
 *   2. Sparse Flash Attention that gathers the selected entries of a paged FP8 MLA
 *      latent cache and runs online-softmax attention over them (dsa_sparse_attn).
 * Two cache writers fill the caches (dsa_quant_kv_mxfp8, dsa_quant_kv_fp8; dsa_quant_kv
 * runs both in one launch), and dsa_decode_step runs a whole decode step in one call.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller (for instance memory
 *   allocated by torch).  The library never allocates, frees or keeps them.
 * - `stream` is a cudaStream_t passed as void*; NULL means the legacy default stream.
 *   Work is enqueued asynchronously on it; no entry point synchronises except
 *   dsa_device_status.
 * - Return value: DSA_OK (0) or a negative DSA_ERR_* code.  On error nothing was
 *   launched and dsa_last_error() describes the problem.  Errors found on the device
 *   (page ids or positions out of range, rows of one group in different sequences, a
 *   bounded wait that ran out) are recorded in a device status word instead of faulting;
 *   read it with dsa_device_status.
 * - Pages: both caches use 64-token pages and share one page table.  A token at
 *   position p of sequence b lives in physical page page_table[b * max_pages + p / 64],
 *   row p % 64; its cache "slot" is page * 64 + p % 64.
 * - Positions are logical positions inside the sequence (0-based).
 * - Per device, the library looks up the device addresses of its own device-side words
 *   (the status word, the scratch array of dsa_sparse_attn_noalloc) and queries the
 *   multiprocessor count once, then keeps them for the life of the process.  A call
 *   after cudaDeviceReset (or any teardown of the device's primary context) would use
 *   stale addresses: the library must not outlive a reset of a device it has used.
 *
 * Cache layouts (bytes)
 * ---------------------
 * Indexer K-cache, one 8448-byte block per physical page:
 *     [0, 8192)     E4M3 codes, row-major [64 tokens][128 dims]
 *     [8192, 8448)  E8M0 group scales, [64 tokens][4 groups of 32 dims]
 * MLA latent KV-cache, one 608-byte record per token (38912 bytes per page):
 *     [0, 576)      E4M3 codes of the 576 latent dims (512 "nope" + 64 "rope")
 *     [576, 596)    five fp32 scales, one per tile [0,128) [128,256) [256,384)
 *                   [384,512) [512,576)
 *     [596, 608)    zero padding (keeps records 32-byte aligned)
 */
#ifndef DSA_GB300_H
#define DSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_PAGE_SIZE 64
#define DSA_INDEX_DIM 128
#define DSA_LATENT_DIM 576
#define DSA_V_DIM 512
#define DSA_KCACHE_PAGE_BYTES 8448
#define DSA_KVCACHE_TOKEN_BYTES 608

enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = -1, /* a pointer, size or alignment the library cannot accept */
  DSA_ERR_UNSUPPORTED = -2, /* a valid request outside what the kernels implement */
  DSA_ERR_CUDA = -3,        /* a CUDA runtime call or kernel launch failed */
  DSA_ERR_DEVICE = -4       /* dsa_device_status found a recorded device-side error */
};

/* Bits of the device status word (see dsa_device_status). */
enum {
  DSA_STATUS_BAD_PAGE = 1,      /* page id outside [0, num_pages) or slot outside the cache */
  DSA_STATUS_BAD_SEQ = 2,       /* q_seq outside [0, n_seq) or a group spans two sequences */
  DSA_STATUS_BAD_LEN = 4,       /* seq_len outside [0, max_ctx] */
  DSA_STATUS_BAD_INDEX = 8,     /* Top-K index outside the row's sequence */
  DSA_STATUS_TIMEOUT = 16,      /* a bounded wait inside a kernel gave up */
  DSA_STATUS_NAN_SCORE = 32,    /* an indexer score was NaN (ranked below every other score) */
  DSA_STATUS_INTERNAL = 64      /* a kernel found its shared memory misaligned and did nothing */
};

/*
 * dsa_quant_kv_mxfp8 -- write indexer keys into the paged MXFP8 K-cache.
 * Follows "Kimi K3.1 Pro Inference Acceleration: Day0 Optimization on Heterogeneous AI
 * Hardware", section "Full MXFP8 Quantization with Per-Group Dynamic Scaling for LI":
 * E4M3 elements, one E8M0 scale per 32 elements.  Scale rule (OCP MX): shared exponent
 * e = floor(log2(amax)) - 8 clamped to [-127, 127], code e + 127; elements are
 * x * 2^-e rounded to nearest even and saturated to +-448; a zero group gets code 127
 * and zero codes.
 *   k_bf16        [n_tokens][128] bfloat16, row-major, 16-byte aligned.
 *   slot_mapping  [n_tokens] int64 slot of each token; a negative slot skips the token.
 *   k_cache       num_slots / 64 pages of DSA_KCACHE_PAGE_BYTES, 16-byte aligned.
 *   num_slots     cache capacity in tokens (a multiple of 64).
 * Slots >= num_slots are skipped and flag DSA_STATUS_BAD_PAGE.
 */
int dsa_quant_kv_mxfp8(const void* k_bf16, const int64_t* slot_mapping, int32_t n_tokens,
                       uint8_t* k_cache, int64_t num_slots, void* stream);

/*
 * dsa_quant_kv_fp8 -- write MLA latent rows into the paged FP8 KV-cache.
 * Follows the same page, section "FP8 KVCache with Per-Token-Head-Tile Quantization for
 * SFA": one fp32 scale per 128-element tile of each token.  Rule: scale =
 * fp32(amax / 448); codes are the exact quotient x / scale rounded once to E4M3 (nearest
 * even, saturating); a zero tile gets scale 0 and zero codes.
 *   kv_bf16       [n_tokens][576] bfloat16, row-major, 16-byte aligned.
 *   slot_mapping  [n_tokens] int64 (negative = skip), as above.
 *   kv_cache      num_slots records of DSA_KVCACHE_TOKEN_BYTES, 16-byte aligned.
 */
int dsa_quant_kv_fp8(const void* kv_bf16, const int64_t* slot_mapping, int32_t n_tokens,
                     uint8_t* kv_cache, int64_t num_slots, void* stream);

/*
 * dsa_quant_kv -- both writers above for the same tokens in one launch: token i's key
 * k_bf16[i] goes to the MXFP8 K-cache and its latent row kv_bf16[i] to the FP8 KV-cache,
 * both at slot_mapping[i] (the two caches share one page table).  The codes and scales are
 * exactly those of dsa_quant_kv_mxfp8 followed by dsa_quant_kv_fp8; a decode step uses it
 * to write its new tokens with one kernel before the indexer.  The pages give the two
 * formats, not this pairing.
 *   k_bf16, kv_bf16, slot_mapping   as for the two writers above (same n_tokens).
 *   k_cache, kv_cache               both hold at least num_slots slots.
 * Errors and skipped slots as for the two writers.
 */
int dsa_quant_kv(const void* k_bf16, const void* kv_bf16, const int64_t* slot_mapping, int32_t n_tokens,
                 uint8_t* k_cache, uint8_t* kv_cache, int64_t num_slots, void* stream);

/*
 * dsa_indexer_topk -- fused Lightning Indexer + Top-K over the paged MXFP8 K-cache.
 * Follows "Deep Dive into Sparse Attention ..." section 2.1 (score, weighting and Top-K
 * fused in one kernel that reads the paged K-cache directly) and "Kimi K3.1 Pro Inference
 * Acceleration ..." section "Lightning Indexer Three-Stream Coordination".  For query row
 * t of sequence b = q_seq[t] at position q_pos[t], every position p < min(q_pos[t] + 1,
 * seq_lens[b]) is scored
 *     score[t, p] = sum_h w[t, h] * max(0, q_hat[t, h] . k_hat[p])
 * where q_hat is the MXFP8 quantisation of q (done on chip, same rule as
 * dsa_quant_kv_mxfp8) and k_hat the cached keys; the K highest scores are kept, equal
 * scores going to the lower position.  No score matrix is written to memory.
 *   q_bf16      [n_q][h_i][128] bfloat16 indexer queries, 16-byte aligned.
 *   w           [n_q][h_i] fp32 head weights.
 *   h_i         indexer heads, 1..64, with q_group * h_i <= 256.
 *   q_group     1..4 consecutive query rows that share one sequence and are scored in
 *               one pass over its pages (2 for two-token MTP decode); n_q % q_group == 0.
 *   k_cache     the MXFP8 K-cache (layout above); num_pages pages.
 *   page_table  [n_seq][max_pages] int32 physical page ids.
 *   seq_lens    [n_seq] int32, each in [0, max_ctx].
 *   q_seq, q_pos [n_q] int32.
 *   max_ctx     host-side upper bound of seq_lens (sizes the on-chip score buffer);
 *               1..262144.
 *   topk        K, 1..2048.
 *   out_idx     [n_q][topk] int32: the selected positions in no particular order,
 *               -1 in the unused tail when a row has fewer than K selectable positions.
 *   out_scores  nullable [n_q][topk] fp32: the score of each selected position (-inf
 *               where out_idx is -1).
 */
int dsa_indexer_topk(const void* q_bf16, const float* w, int32_t n_q, int32_t h_i,
                     int32_t q_group, const uint8_t* k_cache, int64_t num_pages,
                     const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                     const int32_t* q_seq, const int32_t* q_pos, int32_t n_seq,
                     int32_t max_ctx, int32_t topk, int32_t* out_idx, float* out_scores,
                     void* stream);

/*
 * dsa_indexer_scores -- the same scores as dsa_indexer_topk, written out in full
 * (a checking aid: the fused entry point never writes them).
 *   out_scores  [n_q][max_ctx] fp32; positions a row may not select get -inf.
 * Other arguments as dsa_indexer_topk (topk is not used).
 */
int dsa_indexer_scores(const void* q_bf16, const float* w, int32_t n_q, int32_t h_i,
                       int32_t q_group, const uint8_t* k_cache, int64_t num_pages,
                       const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                       const int32_t* q_seq, const int32_t* q_pos, int32_t n_seq,
                       int32_t max_ctx, float* out_scores, void* stream);

/*
 * dsa_sparse_attn_workspace_size -- bytes of device scratch dsa_sparse_attn needs for
 * these sizes (0 is possible).
 */
size_t dsa_sparse_attn_workspace_size(int32_t n_q, int32_t h_s, int32_t topk);

/*
 * dsa_sparse_attn -- Sparse Flash Attention over the selected latent-cache entries.
 * Follows "Adapting and Optimizing Kimi K3.1 Pro for Long-Sequence Inference" section 2
 * (gather the cache entries named by the previous step's indices) and "Kimi K3.1 Pro
 * Inference Acceleration ..." section "Preserving a Mixed-Precision Path" (BF16 query
 * and output).  Absorbed-MLA decode: each selected position j gives one dequantised
 * latent row kv[j] (576 wide) used as the key, and kv[j][0:512] is the value:
 *     l_j = sm_scale * q[t, h] . kv[j];  o[t, h] = sum_j softmax(l)_j kv[j][0:512]
 *     lse[t, h] = log sum_j exp(l_j)
 * over the entries of topk_idx[t] that are >= 0.  A row with no entry gets o = 0 and
 * lse = -inf.  Entries >= the sequence length flag DSA_STATUS_BAD_INDEX and are skipped.
 *   q_bf16     [n_q][h_s][576] bfloat16, 16-byte aligned.
 *   h_s        SFA heads, 1..128.
 *   kv_cache   the FP8 latent cache (layout above), num_pages pages.
 *   page_table, max_pages, seq_lens, q_seq, n_seq: as dsa_indexer_topk.
 *   topk_idx   [n_q][topk] int32 positions (for instance dsa_indexer_topk's out_idx).
 *   out_bf16   [n_q][h_s][512] bfloat16.
 *   out_lse    nullable [n_q][h_s] fp32.
 *   workspace  device scratch of at least dsa_sparse_attn_workspace_size bytes,
 *              256-byte aligned (may be NULL when that size is 0).  Its contents need
 *              not be initialised and are not meaningful afterwards.
 */
int dsa_sparse_attn(const void* q_bf16, int32_t n_q, int32_t h_s, const uint8_t* kv_cache,
                    int64_t num_pages, const int32_t* page_table, int32_t max_pages,
                    const int32_t* seq_lens, const int32_t* q_seq, int32_t n_seq,
                    const int32_t* topk_idx, int32_t topk, float sm_scale, void* out_bf16,
                    float* out_lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * dsa_decode_step -- one decode step of a DSA layer in one call: dsa_quant_kv for the
 * step's new tokens, then dsa_indexer_topk, then dsa_sparse_attn over its out_idx, on
 * `stream`, with the results each of those calls gives.  The pages describe the two
 * stages and the cache writes ("Kimi K3.1 Pro Inference Acceleration ...", section
 * "Lightning Indexer Three-Stream Coordination": the cache write runs alongside the
 * indexer prolog), not this packaging.
 *   When n_new == n_q, new token i must be query row i's own token: slot_mapping[i] is
 *   the slot of position q_pos[i] of sequence q_seq[i] (a decode step's usual case).  The
 *   indexer kernel then writes the tokens itself -- each in the CTA that scans its page,
 *   before it loads that page -- and no writer kernel runs.  A slot_mapping[i] that is not
 *   row i's own slot flags DSA_STATUS_BAD_PAGE (the token is still written there).
 *   Otherwise the writer kernel runs first; the indexer reads its queries, weights,
 *   sequence information and page table while the writer is still running, and only its
 *   K-cache copies wait for the writer.
 *   k_new_bf16, kv_new_bf16, slot_mapping, n_new   as for dsa_quant_kv (n_new may be 0:
 *                        nothing is written, and the indexer waits as usual).
 *   k_cache, kv_cache    both caches, num_pages pages each (slots 0 .. 64 num_pages - 1).
 *   page_table .. q_group, q_idx_bf16, w, h_i, topk, out_idx   as for dsa_indexer_topk
 *                        (out_scores is not produced).
 *   q_sfa_bf16, h_s, sm_scale, out_bf16, out_lse, workspace, workspace_bytes   as for
 *                        dsa_sparse_attn (topk_idx is out_idx).
 * Every argument is checked before anything is launched; errors as for the three calls.
 */
int dsa_decode_step(const void* k_new_bf16, const void* kv_new_bf16, const int64_t* slot_mapping, int32_t n_new,
                    uint8_t* k_cache, uint8_t* kv_cache, int64_t num_pages, const int32_t* page_table,
                    int32_t max_pages, const int32_t* seq_lens, int32_t n_seq, int32_t max_ctx, int32_t n_q,
                    const int32_t* q_seq, const int32_t* q_pos, int32_t q_group, const void* q_idx_bf16,
                    const float* w, int32_t h_i, int32_t topk, int32_t* out_idx, const void* q_sfa_bf16,
                    int32_t h_s, float sm_scale, void* out_bf16, float* out_lse, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * dsa_sparse_attn_noalloc -- dsa_sparse_attn for callers that cannot allocate device
 * memory.  The pages have no counterpart: this is a convenience of this library.
 * Some callers have no allocator they may use for the split-merge workspace -- code that
 * runs under a framework owning every allocation, or on a path where an allocation call
 * would synchronise the device.  This variant keeps that workspace in one fixed array of
 * DSA_NOALLOC_SCRATCH_BYTES inside the library, reserved on every GPU that loads the
 * library until the process exits; it allocates nothing and frees nothing.
 *   Arguments, outputs and errors are those of dsa_sparse_attn, without the workspace.
 *   Sizes whose workspace (dsa_sparse_attn_workspace_size) exceeds
 *   DSA_NOALLOC_SCRATCH_BYTES are rejected with DSA_ERR_UNSUPPORTED and a message.
 *   The first call on a device looks up the array's device address with that device
 *   current; make that first call before any stream capture.
 *   Every call on a device shares the array and it keeps the last call's contents (no
 *   part of it needs to start at zero).  Calls whose kernels overlap on the GPU -- on
 *   different streams, or from different threads -- race on it: serialise them.
 */
#define DSA_NOALLOC_SCRATCH_BYTES (40u * 1024u * 1024u)
int dsa_sparse_attn_noalloc(const void* q_bf16, int32_t n_q, int32_t h_s, const uint8_t* kv_cache,
                            int64_t num_pages, const int32_t* page_table, int32_t max_pages,
                            const int32_t* seq_lens, const int32_t* q_seq, int32_t n_seq,
                            const int32_t* topk_idx, int32_t topk, float sm_scale, void* out_bf16,
                            float* out_lse, void* stream);

/*
 * dsa_device_status -- synchronise `stream`, return the device status word (an OR of
 * DSA_STATUS_* bits recorded by kernels since the last call on this device) and clear
 * it.  Returns a negative DSA_ERR_CUDA if the synchronisation itself failed.
 */
int dsa_device_status(void* stream);

/*
 * Context parallelism.  "Deep Dive into Sparse Attention ..." section 3 and "Adapting and
 * Optimizing Kimi K3.1 Pro for Long-Sequence Inference" section 4 shard the context of a
 * long sequence over devices.  Each device runs dsa_indexer_topk on its shard (a
 * page-aligned range of positions [lo, hi), seen as a sequence of its own: the page-table
 * slice, seq_len hi - lo, q_pos - lo), keeping its local Top-K with scores; the devices
 * exchange those candidates once; dsa_topk_merge turns them into the global Top-K; each
 * device runs dsa_sparse_attn over the selected entries in its shard; the devices
 * exchange (o, lse) once more; dsa_lse_combine gives the output.  Both exchanges are the
 * caller's (for instance an all-gather); the result equals the single-device path.
 */

/*
 * dsa_topk_merge -- the K highest of several parts' candidates, per query row.
 *   cand_idx      [n_parts][n_q][k_in] int32 part-local positions, -1 = empty.
 *   cand_scores   [n_parts][n_q][k_in] fp32 their scores.
 *   part_offsets  nullable [n_parts][n_q] int32 added to part p's positions of row t
 *                 (a shard's first position); null means 0.
 *   topk          K.  n_parts * k_in <= 16384.
 *   out_idx       [n_q][topk] int32 global positions ordered by score (highest first),
 *                 equal scores by lower position; -1 after the last real candidate.
 *   out_scores    nullable [n_q][topk] fp32 their scores (-inf where out_idx is -1).
 *   local_lo, local_hi, out_local   all null, or all given: [n_q] int32 bounds of this
 *                 device's shard and [n_q][topk] int32 out_idx - local_lo where out_idx lies
 *                 in [local_lo, local_hi), else -1 (the selected entries this device holds,
 *                 as positions of its shard, ready for dsa_sparse_attn).
 * NaN scores rank below every other score.  A merged position outside int32 flags
 * DSA_STATUS_BAD_INDEX and is dropped.
 */
int dsa_topk_merge(const int32_t* cand_idx, const float* cand_scores, const int32_t* part_offsets, int32_t n_parts,
                   int32_t n_q, int32_t k_in, int32_t topk, int32_t* out_idx, float* out_scores,
                   const int32_t* local_lo, const int32_t* local_hi, int32_t* out_local, void* stream);

/*
 * dsa_lse_combine -- combine attention outputs over disjoint sets of entries.
 *   o_parts    [n_parts][n_q][h][512] bfloat16, each part normalised over its own entries
 *              (as dsa_sparse_attn writes it), 8-byte aligned.
 *   lse_parts  [n_parts][n_q][h] fp32 each part's log-sum-exp (natural log; -inf = the part
 *              had no entry).
 *   out_bf16   [n_q][h][512] bfloat16: sum_p exp(lse_p - L) o_p, L = log sum_p exp(lse_p).
 *   out_lse    nullable [n_q][h] fp32 L.
 * The softmax over a union of disjoint sets is this weighting of the softmaxes over the sets.
 */
int dsa_lse_combine(const void* o_parts, const float* lse_parts, int32_t n_parts, int32_t n_q, int32_t h,
                    void* out_bf16, float* out_lse, void* stream);

/*
 * dsa_test_stall_indexer -- a testing aid for the kernels' bounded waits; not for
 * production use.  Every wait inside a kernel on an mbarrier gives up after a limit
 * (about one second), sets DSA_STATUS_TIMEOUT and lets the kernel finish instead of
 * hanging.  With wait_limit_us > 0, every indexer launch that follows in this process
 * (dsa_indexer_topk, dsa_indexer_scores, dsa_decode_step) uses that limit, and its
 * copy-issuing lanes stop before their first copy, as a stalled producer would.  The
 * consumers' waits then run out: the kernel sets DSA_STATUS_TIMEOUT, skips the rest of its
 * work, waits for its own copies and tensor-core products in flight, frees its tensor
 * memory and returns; its rows come back as -1 (no position scored).  0 restores normal
 * operation.  Returns DSA_ERR_INVALID_ARG outside 0..10000000.
 */
int dsa_test_stall_indexer(int32_t wait_limit_us);

/* dsa_last_error -- message for the last non-zero return on this host thread. */
const char* dsa_last_error(void);

/* dsa_version -- ABI version (major * 100 + minor). */
int dsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_H */
