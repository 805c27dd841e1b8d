// Sparse Flash Attention over the selected entries of the paged FP8 MLA latent cache.
//
// "Deep Dive into Sparse Attention and Engineering Optimizations for Efficient Inference
// in Kimi K3.1 Pro", section 1 (attention only over the selected positions) and "Adapting
// and Optimizing Kimi K3.1 Pro for Long-Sequence Inference", section 2 (gather of the
// cache entries named by the indexer's indices).  Absorbed MLA: the dequantised 576-wide
// latent row of a selected position is the key, its first 512 entries the value.
//
// This version runs on the CUDA cores: one CTA per (query row, 16 heads) walks the
// selected entries in tiles of 32, gathers and dequantises each tile into shared
// memory (code * tile scale, fp32), and keeps an online softmax with the output
// accumulator in registers.

#include <cfloat>

#include "dsa_common.cuh"
#include "dsa_launch.h"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kHeads = 16;       // heads per CTA
constexpr int kTok = 32;         // selected entries per tile
constexpr int kRow = kLatent + 4;  // padded fp32 row stride of the kv tile (bank spread)

struct SfaSmem {
  float q[kHeads][kLatent];
  float kv[kTok][kRow];
  float p[kHeads][kTok];
  float alpha[kHeads];
  float m[kHeads];
  float l[kHeads];
  const uint8_t* rec[kTok];
};

__global__ void __launch_bounds__(kThreads)
sfa_cuda_core_kernel(SfaArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SfaSmem& sm = *reinterpret_cast<SfaSmem*>(smem_raw);
  const int t = blockIdx.x;
  const int h0 = blockIdx.y * kHeads;
  const int nh = min(kHeads, a.h_s - h0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const int seq = a.q_seq[t];
  const bool seq_ok = seq >= 0 && seq < a.n_seq;
  if (!seq_ok && tid == 0) flag(a.status, DSA_STATUS_BAD_SEQ);
  const int L = seq_ok ? a.seq_lens[seq] : 0;
  const int32_t* ptab = a.page_table + static_cast<size_t>(seq_ok ? seq : 0) * a.max_pages;

  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + (static_cast<size_t>(t) * a.h_s + h0) * kLatent;
  for (int i = tid; i < kHeads * kLatent; i += kThreads) {
    const int h = i / kLatent;
    sm.q[h][i % kLatent] = (h < nh) ? __bfloat162float(q[i]) * a.sm_scale : 0.f;
  }
  if (tid < kHeads) { sm.m[tid] = -INFINITY; sm.l[tid] = 0.f; }

  // output accumulator: thread owns dims 2*tid, 2*tid+1 of all 16 heads
  float acc[kHeads][2];
#pragma unroll
  for (int h = 0; h < kHeads; ++h) acc[h][0] = acc[h][1] = 0.f;

  const int32_t* idx = a.idx + static_cast<size_t>(t) * a.topk;
  for (int j0 = 0; j0 < a.topk; j0 += kTok) {
    __syncthreads();
    if (tid < kTok) {
      const int j = j0 + tid;
      const uint8_t* rec = nullptr;
      if (j < a.topk) {
        const int p = idx[j];
        if (p >= 0) {
          if (p >= L || p / kPage >= a.max_pages) {
            flag(a.status, DSA_STATUS_BAD_INDEX);
          } else {
            const int page = ptab[p / kPage];
            if (page < 0 || page >= a.num_pages) flag(a.status, DSA_STATUS_BAD_PAGE);
            else rec = a.kv_cache + (static_cast<int64_t>(page) * kPage + p % kPage) * kKvTokBytes;
          }
        }
      }
      sm.rec[tid] = rec;
    }
    __syncthreads();
    // gather + dequantise: 32 entries x 144 words of 4 codes
    for (int e = tid; e < kTok * (kLatent / 4); e += kThreads) {
      const int j = e / (kLatent / 4), c4 = e % (kLatent / 4);
      const uint8_t* rec = sm.rec[j];
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (rec) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(rec + 4 * c4);
        const float s = *reinterpret_cast<const float*>(rec + kKvScaleOff + 4 * ((4 * c4) / 128));
        e4m3x4_to_f32(w, v);
        v[0] *= s; v[1] *= s; v[2] *= s; v[3] *= s;
      }
      *reinterpret_cast<float4*>(&sm.kv[j][4 * c4]) = make_float4(v[0], v[1], v[2], v[3]);
    }
    __syncthreads();
    // logits: 16 heads x 32 entries; thread -> (head, 2 entries)
    {
      const int h = tid >> 4, jj = tid & 15;
      float s0 = 0.f, s1 = 0.f;
      const float* qh = sm.q[h];
      const float* k0 = sm.kv[jj];
      const float* k1 = sm.kv[jj + 16];
      for (int d = 0; d < kLatent; d += 4) {
        const float4 qq = *reinterpret_cast<const float4*>(qh + d);
        const float4 a0 = *reinterpret_cast<const float4*>(k0 + d);
        const float4 a1 = *reinterpret_cast<const float4*>(k1 + d);
        s0 = fmaf(qq.x, a0.x, fmaf(qq.y, a0.y, fmaf(qq.z, a0.z, fmaf(qq.w, a0.w, s0))));
        s1 = fmaf(qq.x, a1.x, fmaf(qq.y, a1.y, fmaf(qq.z, a1.z, fmaf(qq.w, a1.w, s1))));
      }
      sm.p[h][jj] = sm.rec[jj] ? s0 : -INFINITY;
      sm.p[h][jj + 16] = sm.rec[jj + 16] ? s1 : -INFINITY;
    }
    __syncthreads();
    // online softmax: warp w handles heads 2w, 2w+1; lane = entry
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = 2 * warp + hh;
      const float s = sm.p[h][lane];
      float mx = s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_old = sm.m[h];
      const float m_new = fmaxf(m_old, mx);
      const float pj = (m_new == -INFINITY) ? 0.f : expf(s - m_new);
      float sum = pj;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      __syncwarp();
      sm.p[h][lane] = pj;
      if (lane == 0) {
        const float al = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
        sm.alpha[h] = al;
        sm.m[h] = m_new;
        sm.l[h] = sm.l[h] * al + sum;
      }
    }
    __syncthreads();
    // O = alpha * O + P V
#pragma unroll
    for (int h = 0; h < kHeads; ++h) {
      const float al = sm.alpha[h];
      float o0 = acc[h][0] * al, o1 = acc[h][1] * al;
#pragma unroll 8
      for (int j = 0; j < kTok; ++j) {
        const float pj = sm.p[h][j];
        const float2 v = *reinterpret_cast<const float2*>(&sm.kv[j][2 * tid]);
        o0 = fmaf(pj, v.x, o0);
        o1 = fmaf(pj, v.y, o1);
      }
      acc[h][0] = o0;
      acc[h][1] = o1;
    }
  }
  __syncthreads();
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (static_cast<size_t>(t) * a.h_s + h0) * kVDim;
  for (int h = 0; h < nh; ++h) {
    const float l = sm.l[h];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    *reinterpret_cast<__nv_bfloat162*>(out + h * kVDim + 2 * tid) =
        __floats2bfloat162_rn(acc[h][0] * inv, acc[h][1] * inv);
  }
  if (a.out_lse && tid < nh) {
    const float l = sm.l[tid];
    a.out_lse[static_cast<size_t>(t) * a.h_s + h0 + tid] = l > 0.f ? sm.m[tid] + logf(l) : -INFINITY;
  }
}

}  // namespace

size_t sfa_workspace_bytes(int, int, int) { return 0; }

cudaError_t launch_sfa(const SfaArgs& a, cudaStream_t s, const char** err) {
  (void)err;
  if (a.n_q == 0) return cudaSuccess;
  const size_t smem = sizeof(SfaSmem);
  cudaError_t e = cudaFuncSetAttribute(sfa_cuda_core_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_q, (a.h_s + kHeads - 1) / kHeads);
  sfa_cuda_core_kernel<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dsa
