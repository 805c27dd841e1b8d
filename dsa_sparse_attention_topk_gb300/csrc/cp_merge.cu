// The two merge steps of context-parallel decoding.
//
// "Deep Dive into Sparse Attention and Engineering Optimizations for Efficient Inference
// in Kimi K3.1 Pro", section 3 ("Introduction of Context Parallelism"), and "Adapting and
// Optimizing Kimi K3.1 Pro for Long-Sequence Inference", section 4: the context of one
// long sequence is sharded over devices; each device scores its shard and keeps its local
// Top-K, the devices exchange those candidates once and merge them into the global Top-K,
// each runs sparse attention over the selected entries it holds, and the partial outputs
// are combined.
//
//   topk_merge_kernel   one CTA per query row: every part's (index, score) candidates,
//                       shifted by the part's offset to global positions, are sorted in
//                       shared memory (bitonic, 64-bit keys: score descending, then position
//                       ascending) and the first K are written, -1 after the last real one.
//                       The same order a stable descending sort of all scores gives.
//   lse_combine_kernel  one CTA per (row, head): the parts' normalised outputs weighted by
//                       exp(lse_p - max lse), and the combined log-sum-exp.

#include <cfloat>
#include <cstdint>

#include "dsa_common.cuh"
#include "dsa_launch.h"

namespace dsa {
namespace {

constexpr int kMergeThreads = 1024;

// 64-bit sort key: order-preserving score key (0 = empty) above the complemented position,
// so that a descending sort puts higher scores first and, among equal scores, lower
// positions first.
__device__ __forceinline__ uint64_t merge_key(int32_t pos, float score) {
  if (pos < 0) return 0ull;
  return (static_cast<uint64_t>(score_key(score)) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(pos));
}

__global__ void __launch_bounds__(kMergeThreads)
topk_merge_kernel(const int32_t* __restrict__ cand_idx, const float* __restrict__ cand_scores,
                  const int32_t* __restrict__ part_offsets, int n_parts, int n_q, int k_in, int topk,
                  int n_pow2, int32_t* __restrict__ out_idx, float* __restrict__ out_scores,
                  const int32_t* __restrict__ local_lo, const int32_t* __restrict__ local_hi,
                  int32_t* __restrict__ out_local, unsigned* status) {
  extern __shared__ uint64_t keys[];  // [n_pow2]
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x;
  const int n = n_parts * k_in;
  bool bad = false;
  for (int i = threadIdx.x; i < n_pow2; i += blockDim.x) {
    uint64_t key = 0ull;
    if (i < n) {
      const int p = i / k_in, c = i - p * k_in;
      const size_t src = (static_cast<size_t>(p) * n_q + t) * k_in + c;
      const int32_t li = cand_idx[src];
      if (li >= 0) {
        const int64_t g = static_cast<int64_t>(li) + (part_offsets ? part_offsets[static_cast<size_t>(p) * n_q + t] : 0);
        if (g < 0 || g > 0x7FFFFFFEll) {
          bad = true;
        } else {
          key = merge_key(static_cast<int32_t>(g), cand_scores[src]);
        }
      }
    }
    keys[i] = key;
  }
  if (bad) flag(status, DSA_STATUS_BAD_INDEX);
  __syncthreads();
  // bitonic sort, descending
  for (int size = 2; size <= n_pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n_pow2 / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));  // index of the pair's lower element
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t a = keys[lo], b = keys[hi];
        if ((a < b) == desc) {
          keys[lo] = b;
          keys[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  const int32_t lo_t = local_lo ? local_lo[t] : 0, hi_t = local_hi ? local_hi[t] : 0;
  for (int s = threadIdx.x; s < topk; s += blockDim.x) {
    const uint64_t key = s < n_pow2 ? keys[s] : 0ull;
    int32_t pos = -1;
    float sc = -INFINITY;
    if (key != 0ull) {
      pos = static_cast<int32_t>(~static_cast<uint32_t>(key & 0xFFFFFFFFull));
      sc = key_score(static_cast<uint32_t>(key >> 32));
    }
    const size_t o = static_cast<size_t>(t) * topk + s;
    out_idx[o] = pos;
    if (out_scores) out_scores[o] = sc;
    if (out_local) out_local[o] = (pos >= lo_t && pos < hi_t) ? pos - lo_t : -1;
  }
}

// o = sum_p w_p o_p / sum_p w_p with w_p = exp(lse_p - M), M = max_p lse_p; a part with
// lse = -inf (nothing selected there) has weight 0; lse = M + log sum_p w_p.
__global__ void __launch_bounds__(128)
lse_combine_kernel(const __nv_bfloat16* __restrict__ o_parts, const float* __restrict__ lse_parts, int n_parts,
                   int n_q, int h, __nv_bfloat16* __restrict__ out, float* __restrict__ out_lse) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x, hh = blockIdx.y;
  float M = -INFINITY;
  for (int p = 0; p < n_parts; ++p) M = fmaxf(M, lse_parts[(static_cast<size_t>(p) * n_q + t) * h + hh]);
  float wsum = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int p = 0; p < n_parts; ++p) {
    const size_t row = (static_cast<size_t>(p) * n_q + t) * h + hh;
    const float l = lse_parts[row];
    const float w = (l == -INFINITY) ? 0.f : expf(l - M);
    wsum += w;
    const uint2 v = *reinterpret_cast<const uint2*>(o_parts + row * kVDim + 4 * threadIdx.x);
    const __nv_bfloat162 v01 = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
    const __nv_bfloat162 v23 = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
    acc[0] += w * __low2float(v01); acc[1] += w * __high2float(v01);
    acc[2] += w * __low2float(v23); acc[3] += w * __high2float(v23);
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat162 r01 = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  __nv_bfloat162 r23 = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
  uint2 r;
  r.x = *reinterpret_cast<uint32_t*>(&r01);
  r.y = *reinterpret_cast<uint32_t*>(&r23);
  *reinterpret_cast<uint2*>(out + (static_cast<size_t>(t) * h + hh) * kVDim + 4 * threadIdx.x) = r;
  if (out_lse && threadIdx.x == 0) out_lse[static_cast<size_t>(t) * h + hh] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

}  // namespace

int topk_merge_pow2(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

cudaError_t launch_topk_merge(const TopkMergeArgs& a, cudaStream_t s) {
  if (a.n_q == 0) return cudaSuccess;
  const int n_pow2 = topk_merge_pow2(a.n_parts * a.k_in);
  const size_t smem = static_cast<size_t>(n_pow2) * sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(topk_merge_kernel, dim3(a.n_q), dim3(kMergeThreads), smem, s, 1, a.cand_idx, a.cand_scores,
                    a.part_offsets, a.n_parts, a.n_q, a.k_in, a.topk, n_pow2, a.out_idx, a.out_scores, a.local_lo,
                    a.local_hi, a.out_local, a.status);
}

cudaError_t launch_lse_combine(const void* o_parts, const float* lse_parts, int n_parts, int n_q, int h, void* out,
                               float* out_lse, cudaStream_t s) {
  if (n_q == 0) return cudaSuccess;
  return launch_pdl(lse_combine_kernel, dim3(n_q, h), dim3(128), 0, s, 1,
                    static_cast<const __nv_bfloat16*>(o_parts), lse_parts, n_parts, n_q, h,
                    static_cast<__nv_bfloat16*>(out), out_lse);
}

}  // namespace dsa
