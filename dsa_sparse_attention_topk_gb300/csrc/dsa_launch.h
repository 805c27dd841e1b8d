// Internal launchers behind the C ABI (argument checking happens in api.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace dsa {

struct IndexerArgs {
  const void* q;             // bf16 [n_q][h_i][128]
  const float* w;            // [n_q][h_i]
  int n_q, h_i, q_group;
  const uint8_t* k_cache;
  int64_t num_pages;
  const int32_t* page_table;
  int max_pages;
  const int32_t* seq_lens;
  const int32_t* q_seq;
  const int32_t* q_pos;
  int n_seq, max_ctx, topk;
  int32_t* out_idx;          // [n_q][topk] or null (scores mode)
  float* out_scores;         // [n_q][topk] or null
  float* out_full;           // [n_q][max_ctx] (scores mode) or null
  unsigned* status;
};

struct SfaArgs {
  const void* q;             // bf16 [n_q][h_s][576]
  int n_q, h_s;
  const uint8_t* kv_cache;
  int64_t num_pages;
  const int32_t* page_table;
  int max_pages;
  const int32_t* seq_lens;
  const int32_t* q_seq;
  int n_seq;
  const int32_t* idx;        // [n_q][topk]
  int topk;
  float sm_scale;
  void* out;                 // bf16 [n_q][h_s][512]
  float* out_lse;            // [n_q][h_s] or null
  void* workspace;
  size_t workspace_bytes;
  unsigned* status;
};

// Each returns cudaSuccess or the launch error; `err` gets a short reason for
// configuration problems detected while planning the launch.
cudaError_t launch_quant_mxfp8(const void* k, const int64_t* slots, int n_tokens, uint8_t* cache,
                               int64_t num_slots, unsigned* status, cudaStream_t s);
cudaError_t launch_quant_fp8(const void* kv, const int64_t* slots, int n_tokens, uint8_t* cache,
                             int64_t num_slots, unsigned* status, cudaStream_t s);
cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t s, const char** err);
cudaError_t launch_sfa(const SfaArgs& a, cudaStream_t s, const char** err);
size_t sfa_workspace_bytes(int n_q, int h_s, int topk);
cudaError_t launch_sfa_noalloc(const SfaArgs& a, cudaStream_t s, const char** err);

}  // namespace dsa
