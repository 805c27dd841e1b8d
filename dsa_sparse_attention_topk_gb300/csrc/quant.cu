// Cache writers: bf16 rows -> paged MXFP8 indexer K-cache and paged FP8 latent KV-cache.
//
// MXFP8 follows "Kimi K3.1 Pro Inference Acceleration: Day0 Optimization on
// Heterogeneous AI Hardware", section "Full MXFP8 Quantization with Per-Group Dynamic
// Scaling for LI" (one scale per 32 elements) with the OCP MX scale rule; the FP8 latent
// cache follows section "FP8 KVCache with Per-Token-Head-Tile Quantization for SFA"
// (one fp32 scale per 128-element tile of each token).
//
// Every writer gives one warp to one token: the reads are 8-byte (k) or 8/4-byte (kv)
// coalesced loads, the amax reductions are warp shuffles, and the writes land in the
// token's cache row.  They are HBM-bound elementwise kernels (a few bytes of math per
// byte moved) and run once per new token, outside the decode hot loop.

#include "dsa_common.cuh"
#include "dsa_launch.h"
#include "quant_tok.cuh"

namespace dsa {
namespace {

constexpr int kWarpsPerBlock = 8;

// Token loop shared by the writers: warp w of block b takes tokens b * 8 + w, + the grid.
#define DSA_FOR_TOKENS(t)                                                                                    \
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5); t < n_tokens;   \
       t += static_cast<int64_t>(gridDim.x) * kWarpsPerBlock)

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
quant_mxfp8_kernel(const __nv_bfloat16* __restrict__ k, const int64_t* __restrict__ slots,
                   int n_tokens, uint8_t* __restrict__ cache, int64_t num_slots,
                   unsigned* status) {
  pdl_launch_dependents();
  pdl_wait();
  DSA_FOR_TOKENS(t) store_k_token(load_k_token(k, slots, t), cache, num_slots, status);
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
quant_fp8_kernel(const __nv_bfloat16* __restrict__ kv, const int64_t* __restrict__ slots,
                 int n_tokens, uint8_t* __restrict__ cache, int64_t num_slots,
                 unsigned* status) {
  pdl_launch_dependents();
  pdl_wait();
  DSA_FOR_TOKENS(t) store_kv_token(load_kv_token(kv, slots, t), cache, num_slots, status);
}

// Both caches of a token in one launch (a decode step writes both before its indexer).
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
quant_both_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ kv,
                  const int64_t* __restrict__ slots, int n_tokens, uint8_t* __restrict__ k_cache,
                  uint8_t* __restrict__ kv_cache, int64_t num_slots, unsigned* status) {
  // dependents are signalled only after the wait: once a dependent starts, every kernel
  // before this one is complete (a decode step's indexer reads its other inputs early)
  pdl_wait();
  pdl_launch_dependents();
  DSA_FOR_TOKENS(t) {
    const KTok kin = load_k_token(k, slots, t);
    const KvTok kvin = load_kv_token(kv, slots, t);
    store_k_token(kin, k_cache, num_slots, status);
    store_kv_token(kvin, kv_cache, num_slots, status);
  }
}

// one warp per token, at most 16 blocks per multiprocessor (the loop strides over the rest)
int grid_for(int n_tokens) {
  DevInfo di;
  const char* why = nullptr;
  const int cap = device_info(&di, &why) ? di.n_sm * 16 : 2048;
  int blocks = (n_tokens + kWarpsPerBlock - 1) / kWarpsPerBlock;
  return blocks < cap ? (blocks < 1 ? 1 : blocks) : cap;
}

}  // namespace

cudaError_t launch_quant_mxfp8(const void* k, const int64_t* slots, int n_tokens, uint8_t* cache,
                               int64_t num_slots, unsigned* status, cudaStream_t s) {
  if (n_tokens == 0) return cudaSuccess;
  return launch_pdl(quant_mxfp8_kernel, dim3(grid_for(n_tokens)), dim3(kWarpsPerBlock * 32), 0, s, 1,
                    static_cast<const __nv_bfloat16*>(k), slots, n_tokens, cache, num_slots, status);
}

cudaError_t launch_quant_fp8(const void* kv, const int64_t* slots, int n_tokens, uint8_t* cache,
                             int64_t num_slots, unsigned* status, cudaStream_t s) {
  if (n_tokens == 0) return cudaSuccess;
  return launch_pdl(quant_fp8_kernel, dim3(grid_for(n_tokens)), dim3(kWarpsPerBlock * 32), 0, s, 1,
                    static_cast<const __nv_bfloat16*>(kv), slots, n_tokens, cache, num_slots, status);
}

cudaError_t launch_quant_both(const void* k, const void* kv, const int64_t* slots, int n_tokens, uint8_t* k_cache,
                              uint8_t* kv_cache, int64_t num_slots, unsigned* status, cudaStream_t s) {
  if (n_tokens == 0) return cudaSuccess;
  return launch_pdl(quant_both_kernel, dim3(grid_for(n_tokens)), dim3(kWarpsPerBlock * 32), 0, s, 1,
                    static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(kv), slots, n_tokens,
                    k_cache, kv_cache, num_slots, status);
}

}  // namespace dsa
