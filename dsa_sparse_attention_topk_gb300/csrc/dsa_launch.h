// Internal launchers behind the C ABI (argument checking happens in api.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace dsa {

// Every kernel of the library is launched with programmatic stream serialization: it may
// begin (set up shared memory, barriers and TMEM) while the previous kernel on the stream
// drains, and it waits for that kernel (griddepcontrol.wait, see dsa_common.cuh) before
// its first global-memory read or write.  cluster_x > 1 adds a cluster dimension.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster_x,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Multiprocessor count and opt-in shared memory per block of the current device, queried
// once per device (under a lock) and cached for the life of the process.  Returns false
// (with `err` set) when there is no current device or its ordinal is 64 or more.
struct DevInfo {
  int n_sm = 0, smem_optin = 0;
};
bool device_info(DevInfo* out, const char** err);

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
  // 1: the previous kernel on the stream is this library's cache writer, which signals its
  // dependents only after its own wait; everything but the K-cache is then complete when
  // the indexer starts, and only the K-cache copies wait for the writer
  int early_inputs = 0;
  // a decode step's new tokens, written by the indexer itself (fuse_writes = 1): token i is
  // query row i's own token (its slot is row i's position in its sequence); its MXFP8 key
  // goes to k_cache and its latent row to kv_cache, both at slot_mapping[i]
  int fuse_writes = 0;
  const void* k_new = nullptr;       // bf16 [n_q][128]
  const void* kv_new = nullptr;      // bf16 [n_q][576]
  const int64_t* slot_mapping = nullptr;
  uint8_t* kv_cache = nullptr;
  int64_t num_slots = 0;
  // testing aid for the bounded waits (dsa_test_stall_indexer): the waits' limit, and 1 to
  // make the copy-issuing lanes stop before their first copy
  uint64_t wait_ns = 1000000000ull;
  int stall_producer = 0;
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

struct TopkMergeArgs {
  const int32_t* cand_idx;      // [n_parts][n_q][k_in] part-local positions, -1 = empty
  const float* cand_scores;     // same layout
  const int32_t* part_offsets;  // [n_parts][n_q] added to a part's positions, or null (0)
  int n_parts, n_q, k_in, topk;
  int32_t* out_idx;             // [n_q][topk]
  float* out_scores;            // [n_q][topk] or null
  const int32_t* local_lo;      // [n_q] or null: with local_hi, the range out_local keeps
  const int32_t* local_hi;
  int32_t* out_local;           // [n_q][topk] or null: out_idx - local_lo inside the range, else -1
  unsigned* status;
};
int topk_merge_pow2(int n);
cudaError_t launch_topk_merge(const TopkMergeArgs& a, cudaStream_t s);
cudaError_t launch_lse_combine(const void* o_parts, const float* lse_parts, int n_parts, int n_q, int h, void* out,
                               float* out_lse, cudaStream_t s);

// Each returns cudaSuccess or the launch error; `err` gets a short reason for
// configuration problems detected while planning the launch.
cudaError_t launch_quant_mxfp8(const void* k, const int64_t* slots, int n_tokens, uint8_t* cache,
                               int64_t num_slots, unsigned* status, cudaStream_t s);
cudaError_t launch_quant_fp8(const void* kv, const int64_t* slots, int n_tokens, uint8_t* cache,
                             int64_t num_slots, unsigned* status, cudaStream_t s);
cudaError_t launch_quant_both(const void* k, const void* kv, const int64_t* slots, int n_tokens, uint8_t* k_cache,
                              uint8_t* kv_cache, int64_t num_slots, unsigned* status, cudaStream_t s);
cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t s, const char** err);
cudaError_t launch_sfa(const SfaArgs& a, cudaStream_t s, const char** err);
size_t sfa_workspace_bytes(int n_q, int h_s, int topk);
cudaError_t launch_sfa_noalloc(const SfaArgs& a, cudaStream_t s, const char** err);

}  // namespace dsa
