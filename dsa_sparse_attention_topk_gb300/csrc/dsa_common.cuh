// Shared device helpers of the DSA kernels: FP8 conversions, order-preserving score
// keys, cluster (DSMEM) primitives and the device status word.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/dsa.h"

namespace dsa {

constexpr int kPage = DSA_PAGE_SIZE;                 // tokens per page
constexpr int kIdxDim = DSA_INDEX_DIM;               // indexer head dim
constexpr int kLatent = DSA_LATENT_DIM;              // MLA latent width (512 + 64)
constexpr int kVDim = DSA_V_DIM;                     // value width
constexpr int kKPageBytes = DSA_KCACHE_PAGE_BYTES;   // 64*128 codes + 64*4 scales
constexpr int kKScaleOff = kPage * kIdxDim;          // offset of the scale block in a page
constexpr int kKvTokBytes = DSA_KVCACHE_TOKEN_BYTES; // 576 codes + 5 fp32 scales + pad
constexpr int kKvScaleOff = kLatent;                 // offset of the scales in a record
constexpr int kKvTiles = 5;                          // 128-wide tiles of a latent row

// ---------------------------------------------------------------------------------
// Status word: kernels OR error bits into it instead of faulting.
__device__ __forceinline__ void flag(unsigned* status, unsigned bits) {
  if (status) atomicOr(status, bits);
}

// ---------------------------------------------------------------------------------
// E4M3 conversions through the hardware cvt instructions.
// Two floats -> two E4M3 codes, round to nearest even, saturating; lo -> byte 0.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes (byte 0, byte 1) -> two fp16 values (exact: E4M3 is a subset of fp16).
__device__ __forceinline__ __half2 e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return *reinterpret_cast<__half2*>(&r);
}

// Four E4M3 codes packed in a uint32 -> four floats (exact).
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t v, float out[4]) {
  float2 a = __half22float2(e4m3x2_to_f16x2(static_cast<uint16_t>(v & 0xFFFFu)));
  float2 b = __half22float2(e4m3x2_to_f16x2(static_cast<uint16_t>(v >> 16)));
  out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
}

// 2^e as a float for e in [-149, 127] (exact; builds the bit pattern directly).
__device__ __forceinline__ float exp2i(int e) {
  if (e >= -126) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
  return __uint_as_float(1u << (e + 149));
}

// OCP MX shared exponent of a group whose largest magnitude is amax (a finite float):
// floor(log2(amax)) - 8 clamped to [-127, 127]; 0 for amax == 0.
__device__ __forceinline__ int mx_shared_exp(float amax) {
  uint32_t bits = __float_as_uint(amax);
  int ef = static_cast<int>((bits >> 23) & 0xFF);
  if (amax == 0.f) return 0;
  if (ef == 0) return -127;            // subnormal amax: floor(log2) <= -127
  int e = ef - 127 - 8;
  return e < -127 ? -127 : e;
}

// ---------------------------------------------------------------------------------
// Score keys: an order-preserving map float -> uint32 (larger score, larger key).
// -0 is folded onto +0 so equal scores get equal keys.  Key 0 marks "not selectable".
// Every NaN, whatever its sign or payload, maps to key 1: below every other score (a
// stable descending sort puts NaN last), so NaN scores are kept only when fewer than K
// others are selectable, lowest positions first.
constexpr uint32_t kNanKey = 1u;
__device__ __forceinline__ uint32_t score_key(float s) {
  if (s != s) return kNanKey;
  s = s + 0.0f;  // -0 -> +0
  uint32_t b = __float_as_uint(s);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
// max(x, 0) that keeps NaN (fmaxf would return 0 for a NaN x).
__device__ __forceinline__ float relu_nan(float x) {
  float y;
  asm("max.NaN.f32 %0, %1, 0f00000000;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float key_score(uint32_t k) {
  uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(b);
}

// ---------------------------------------------------------------------------------
// Thread-block-cluster helpers (distributed shared memory).
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Programmatic dependent launch: let the next kernel on the stream begin launching, and
// wait until the previous kernel has completed and its memory is visible.  Every kernel
// calls pdl_wait() before its first global read or write.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(local)), "r"(rank));
  return out;
}
__device__ __forceinline__ void dsmem_add_u32(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void dsmem_st_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void dsmem_st_v2(uint32_t addr, uint2 v) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" :: "r"(addr), "r"(v.x), "r"(v.y) : "memory");
}
// Store 8 bytes into another CTA's shared memory and count them on that CTA's mbarrier
// (complete-tx): the receiver learns that the data has landed from the barrier alone.
__device__ __forceinline__ void dsmem_st_async_v2(uint32_t addr, uint2 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.u32 [%0], {%1, %2}, [%3];"
               :: "r"(addr), "r"(v.x), "r"(v.y), "r"(bar) : "memory");
}
__device__ __forceinline__ uint4 dsmem_ld_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

}  // namespace dsa
