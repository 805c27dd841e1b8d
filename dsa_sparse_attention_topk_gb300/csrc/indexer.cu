// Fused Lightning Indexer + Top-K over the paged MXFP8 K-cache.
//
// "Deep Dive into Sparse Attention and Engineering Optimizations for Efficient Inference
// in Kimi K3.1 Pro", section 2.1, and "Kimi K3.1 Pro Inference Acceleration: Day0
// Optimization on Heterogeneous AI Hardware", section "Lightning Indexer Three-Stream
// Coordination": relevance scoring, head-weight weighting and Top-K selection run in one
// kernel that reads the paged K-cache directly; the scores stay on chip.
//
//   score[t, p] = sum_h w[t, h] * max(0, q_hat[t, h] . k_hat[p])
//
// Work split: a group of q_group query rows of one sequence is handled by one
// thread-block cluster of C CTAs; CTA r scores the r-th contiguous chunk of the
// sequence's selectable positions (a multiple of 128 positions), keeps the
// order-preserving keys of its chunk in shared memory, and the cluster selects the
// Top-K of each row over distributed shared memory (topk_cluster.cuh).
//
// Scoring (this file): each thread scores one position at a time on the CUDA cores.
// The MXFP8 query is quantised on chip (same OCP MX rule as the cache writer) and kept
// dequantised in shared memory; the page row of the position is loaded with 16-byte
// loads and dequantised in registers.

#include <cfloat>

#include "dsa_common.cuh"
#include "dsa_launch.h"
#include "topk_cluster.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 128;          // chunk granularity (positions)
constexpr int kMaxCluster = 16;

struct IdxSmemHead {
  TopkSmem topk;
  int seq;                       // sequence of the group
  int n_sel[4];                  // selectable positions per row
  int n_max;
};

// Dynamic shared memory: [IdxSmemHead][w: G*H floats][q_hat: G*H*128 floats][keys: G*chunk_cap]
__host__ __device__ inline size_t idx_smem_bytes(int G, int H, int chunk_cap) {
  size_t head = (sizeof(IdxSmemHead) + 15) & ~size_t(15);
  return head + sizeof(float) * ((G * H + 3) & ~3) + sizeof(float) * G * H * kIdxDim +
         sizeof(uint32_t) * size_t(G) * chunk_cap;
}

// MXFP8-quantise one 128-wide bf16 row and return its dequantised values (lane owns
// elements 4*lane .. 4*lane+3).  Same rule as the cache writer.
__device__ __forceinline__ void quant_dequant_row(const __nv_bfloat16* src, float out[4]) {
  const int lane = threadIdx.x & 31;
  const uint2 raw = *reinterpret_cast<const uint2*>(src + 4 * lane);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
  float x[4] = {__low2float(a), __high2float(a), __low2float(b), __high2float(b)};
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = mx_shared_exp(amax);
  const float inv = exp2i(-e), sc = exp2i(e);
  if (amax == 0.f) {
    out[0] = out[1] = out[2] = out[3] = 0.f;
    return;
  }
  const uint32_t c = static_cast<uint32_t>(f32x2_to_e4m3x2(x[0] * inv, x[1] * inv)) |
                     (static_cast<uint32_t>(f32x2_to_e4m3x2(x[2] * inv, x[3] * inv)) << 16);
  float d[4];
  e4m3x4_to_f32(c, d);
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = d[i] * sc;
}

template <int G>
__global__ void __launch_bounds__(kThreads)
indexer_cuda_core_kernel(IndexerArgs a, int chunk_cap) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  IdxSmemHead& hd = *reinterpret_cast<IdxSmemHead*>(smem_raw);
  const size_t head = (sizeof(IdxSmemHead) + 15) & ~size_t(15);
  const int H = a.h_i;
  float* s_w = reinterpret_cast<float*>(smem_raw + head);
  float* s_q = s_w + ((G * H + 3) & ~3);  // 16-byte aligned for the float4 stores
  uint32_t* s_keys = reinterpret_cast<uint32_t*>(s_q + G * H * kIdxDim);

  const int tid = threadIdx.x;
  const int rank = static_cast<int>(cluster_ctarank());
  const int C = static_cast<int>(cluster_nctarank());
  const int group = blockIdx.y;
  const int row0 = group * G;

  topk_init(hd.topk);
  if (tid == 0) {
    int seq = a.q_seq[row0];
    unsigned bad = 0;
    if (seq < 0 || seq >= a.n_seq) { bad |= DSA_STATUS_BAD_SEQ; seq = -1; }
    int L = 0;
    if (seq >= 0) {
      L = a.seq_lens[seq];
      if (L < 0 || L > a.max_ctx) { bad |= DSA_STATUS_BAD_LEN; L = L < 0 ? 0 : a.max_ctx; }
    }
    int n_max = 0;
    for (int j = 0; j < G; ++j) {
      if (a.q_seq[row0 + j] != a.q_seq[row0]) bad |= DSA_STATUS_BAD_SEQ;
      long long n = static_cast<long long>(a.q_pos[row0 + j]) + 1;
      n = n < 0 ? 0 : (n > L ? L : n);
      hd.n_sel[j] = static_cast<int>(n);
      n_max = n > n_max ? static_cast<int>(n) : n_max;
    }
    hd.seq = seq;
    hd.n_max = n_max;
    if (bad && rank == 0) flag(a.status, bad);
  }
  // on-chip MXFP8 quantisation of the group's queries (one warp per row-head)
  for (int rh = tid >> 5; rh < G * H; rh += kThreads / 32) {
    float v[4];
    quant_dequant_row(static_cast<const __nv_bfloat16*>(a.q) +
                          (static_cast<size_t>(row0) * H + rh) * kIdxDim, v);
    *reinterpret_cast<float4*>(s_q + rh * kIdxDim + 4 * (tid & 31)) = make_float4(v[0], v[1], v[2], v[3]);
  }
  for (int i = tid; i < G * H; i += kThreads) s_w[i] = a.w[static_cast<size_t>(row0) * H + i];
  cluster_sync();  // every CTA initialised before any DSMEM traffic

  const int seq = hd.seq;
  const int n_max = hd.n_max;
  int chunk = (n_max + C - 1) / C;
  chunk = (chunk + kTile - 1) / kTile * kTile;
  if (chunk > chunk_cap) chunk = chunk_cap;  // host sizing guarantees this never binds
  const int c0 = rank * chunk;
  const int len = max(0, min(chunk, n_max - c0));

  const int32_t* ptab = a.page_table + static_cast<size_t>(seq < 0 ? 0 : seq) * a.max_pages;
  for (int i = tid; i < len; i += kThreads) {
    const int p = c0 + i;
    const int page = (seq < 0 || p / kPage >= a.max_pages) ? -1 : ptab[p / kPage];
    if (page < 0 || page >= a.num_pages) {
      flag(a.status, DSA_STATUS_BAD_PAGE);
#pragma unroll
      for (int j = 0; j < G; ++j) s_keys[j * chunk_cap + i] = 0u;
      continue;
    }
    const uint8_t* base = a.k_cache + static_cast<int64_t>(page) * kKPageBytes;
    const int r = p % kPage;
    const uint32_t sc4 = *reinterpret_cast<const uint32_t*>(base + kKScaleOff + r * 4);
    float k[kIdxDim];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(base + r * kIdxDim + 16 * c);
      const float gs = exp2i(static_cast<int>((sc4 >> (8 * (c >> 1))) & 0xFF) - 127);
      float t[4];
      e4m3x4_to_f32(v.x, t); k[16 * c + 0] = t[0] * gs; k[16 * c + 1] = t[1] * gs; k[16 * c + 2] = t[2] * gs; k[16 * c + 3] = t[3] * gs;
      e4m3x4_to_f32(v.y, t); k[16 * c + 4] = t[0] * gs; k[16 * c + 5] = t[1] * gs; k[16 * c + 6] = t[2] * gs; k[16 * c + 7] = t[3] * gs;
      e4m3x4_to_f32(v.z, t); k[16 * c + 8] = t[0] * gs; k[16 * c + 9] = t[1] * gs; k[16 * c + 10] = t[2] * gs; k[16 * c + 11] = t[3] * gs;
      e4m3x4_to_f32(v.w, t); k[16 * c + 12] = t[0] * gs; k[16 * c + 13] = t[1] * gs; k[16 * c + 14] = t[2] * gs; k[16 * c + 15] = t[3] * gs;
    }
#pragma unroll
    for (int j = 0; j < G; ++j) {
      uint32_t key = 0u;
      if (p < hd.n_sel[j]) {
        float s = 0.f;
        for (int h = 0; h < H; ++h) {
          const float* q = s_q + (j * H + h) * kIdxDim;
          float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
          for (int d = 0; d < kIdxDim; d += 4) {
            const float4 qq = *reinterpret_cast<const float4*>(q + d);
            d0 = fmaf(qq.x, k[d], d0);
            d1 = fmaf(qq.y, k[d + 1], d1);
            d2 = fmaf(qq.z, k[d + 2], d2);
            d3 = fmaf(qq.w, k[d + 3], d3);
          }
          const float dot = (d0 + d1) + (d2 + d3);
          s = fmaf(s_w[j * H + h], fmaxf(dot, 0.f), s);
        }
        if (a.out_full) {
          a.out_full[static_cast<size_t>(row0 + j) * a.max_ctx + p] = s;
        }
        key = score_key(s);
      }
      s_keys[j * chunk_cap + i] = key;
    }
  }
  __syncthreads();

  if (a.out_idx) {
#pragma unroll 1
    for (int j = 0; j < G; ++j) {
      const size_t row = static_cast<size_t>(row0 + j);
      cluster_topk_row(hd.topk, s_keys + j * chunk_cap, c0, len, hd.n_sel[j], a.topk,
                       a.out_idx + row * a.topk, a.out_scores ? a.out_scores + row * a.topk : nullptr);
    }
  }
  cluster_sync();  // no CTA leaves while its shared memory may still be addressed
}

__global__ void fill_kernel(float* p, size_t n, float v) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    p[i] = v;
}

template <int G>
cudaError_t launch_g(const IndexerArgs& a, cudaStream_t s, const char** err) {
  int dev = 0;
  cudaGetDevice(&dev);
  int n_sm = 0, smem_optin = 0;
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const int n_groups = a.n_q / G;
  // smallest power-of-two cluster whose per-CTA score buffer fits, then widen while
  // the grid still fits on the GPU in one wave
  int C = 1;
  auto cap_for = [&](int c) {
    int chunk = (a.max_ctx + c - 1) / c;
    return (chunk + kTile - 1) / kTile * kTile;
  };
  while (C < kMaxCluster && idx_smem_bytes(G, a.h_i, cap_for(C)) > static_cast<size_t>(smem_optin)) C *= 2;
  while (C < kMaxCluster && static_cast<long long>(n_groups) * C * 2 <= n_sm) C *= 2;
  const int chunk_cap = cap_for(C);
  const size_t smem = idx_smem_bytes(G, a.h_i, chunk_cap);
  if (smem > static_cast<size_t>(smem_optin)) {
    *err = "indexer: max_ctx too large for the on-chip score buffer";
    return cudaErrorInvalidValue;
  }
  auto kern = indexer_cuda_core_kernel<G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  if (a.out_full) {
    const size_t n = static_cast<size_t>(a.n_q) * a.max_ctx;
    fill_kernel<<<1024, 256, 0, s>>>(a.out_full, n, -INFINITY);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, n_groups, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, chunk_cap);
}

}  // namespace

cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t s, const char** err) {
  if (a.n_q == 0) return cudaSuccess;
  switch (a.q_group) {
    case 1: return launch_g<1>(a, s, err);
    case 2: return launch_g<2>(a, s, err);
    case 3: return launch_g<3>(a, s, err);
    case 4: return launch_g<4>(a, s, err);
    default: *err = "indexer: q_group must be 1..4"; return cudaErrorInvalidValue;
  }
}

}  // namespace dsa
