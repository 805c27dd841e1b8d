// One-warp-per-token cache writers (device functions), shared by the writer kernels and by
// the indexer of a decode step, which writes the step's new tokens itself.
//
// MXFP8 follows "Kimi K3.1 Pro Inference Acceleration: Day0 Optimization on
// Heterogeneous AI Hardware", section "Full MXFP8 Quantization with Per-Group Dynamic
// Scaling for LI" (one scale per 32 elements) with the OCP MX scale rule; the FP8 latent
// cache follows section "FP8 KVCache with Per-Token-Head-Tile Quantization for SFA"
// (one fp32 scale per 128-element tile of each token).
#pragma once

#include "dsa_common.cuh"

namespace dsa {

// One warp writes token t's indexer key: 128 values, four MXFP8 groups of 32 (group =
// lane / 8, four values per lane).  The loads are issued first (load_k_token), so that a
// caller writing both caches can have every load of a token in flight at once.
struct KTok {
  uint2 raw;     // this lane's four values (dims 4 lane ..)
  int64_t slot;
};
__device__ __forceinline__ KTok load_k_token(const __nv_bfloat16* __restrict__ k, const int64_t* __restrict__ slots,
                                             int64_t t) {
  const int lane = threadIdx.x & 31;
  return KTok{*reinterpret_cast<const uint2*>(k + t * kIdxDim + 4 * lane), slots[t]};
}
__device__ __forceinline__ void store_k_token(const KTok& in, uint8_t* __restrict__ cache, int64_t num_slots,
                                              unsigned* status) {
  const int lane = threadIdx.x & 31;
  const int64_t slot = in.slot;
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (lane == 0) flag(status, DSA_STATUS_BAD_PAGE);
    return;
  }
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&in.raw.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&in.raw.y);
  float x[4] = {__low2float(a), __high2float(a), __low2float(b), __high2float(b)};
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = mx_shared_exp(amax);
  const float inv = exp2i(-e);  // exact power of two: x * inv is exact
  uint32_t codes = 0;
  if (amax > 0.f) {
    codes = static_cast<uint32_t>(f32x2_to_e4m3x2(x[0] * inv, x[1] * inv)) |
            (static_cast<uint32_t>(f32x2_to_e4m3x2(x[2] * inv, x[3] * inv)) << 16);
  }
  uint8_t* page = cache + (slot / kPage) * kKPageBytes;
  const int row = static_cast<int>(slot % kPage);
  *reinterpret_cast<uint32_t*>(page + row * kIdxDim + 4 * lane) = codes;
  if ((lane & 7) == 0) page[kKScaleOff + row * 4 + (lane >> 3)] = static_cast<uint8_t>(e + 127);
}

// |x| / s rounded to the nearest float and then nudged to "round to odd" when inexact:
// converting the result to E4M3 with round-to-nearest-even then gives the correctly
// rounded E4M3 value of the exact quotient (Boldo & Melquiond, "Emulation of FMA and
// correctly rounded sums: proved algorithms using rounding to odd", 2008: rounding to
// odd with p+2 or more bits followed by round-to-nearest is a correct rounding).
__device__ __forceinline__ float quotient_round_to_odd(float x, float s) {
  const float a = fabsf(x);
  const float q = __fdiv_rn(a, s);
  const float r = __fmaf_rn(-q, s, a);  // exact remainder a - q*s
  uint32_t qb = __float_as_uint(q);
  if (r != 0.f && (qb & 1u) == 0u) qb += (r > 0.f) ? 1u : 0xFFFFFFFFu;
  return copysignf(__uint_as_float(qb), x);
}

// One warp writes token t's latent row: four 128-wide tiles (four values per lane) and the
// 64-wide rope tile (two per lane), each with its fp32 scale; loads first, as above.
struct KvTok {
  uint2 raws[4];           // this lane's four values of each full tile
  __nv_bfloat162 rope;     // this lane's two rope values
  int64_t slot;
};
__device__ __forceinline__ KvTok load_kv_token(const __nv_bfloat16* __restrict__ kv, const int64_t* __restrict__ slots,
                                               int64_t t) {
  const int lane = threadIdx.x & 31;
  const __nv_bfloat16* src = kv + t * kLatent;
  KvTok in;
#pragma unroll
  for (int tile = 0; tile < 4; ++tile) in.raws[tile] = *reinterpret_cast<const uint2*>(src + tile * 128 + 4 * lane);
  in.rope = *reinterpret_cast<const __nv_bfloat162*>(src + 512 + 2 * lane);
  in.slot = slots[t];
  return in;
}
__device__ __forceinline__ void store_kv_token(const KvTok& in, uint8_t* __restrict__ cache, int64_t num_slots,
                                               unsigned* status) {
  const int lane = threadIdx.x & 31;
  const int64_t slot = in.slot;
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (lane == 0) flag(status, DSA_STATUS_BAD_PAGE);
    return;
  }
  uint8_t* rec = cache + slot * kKvTokBytes;
  float scales[kKvTiles];
#pragma unroll
  for (int tile = 0; tile < 4; ++tile) {  // four full 128-wide tiles: 4 elements per lane
    const uint2 raw = in.raws[tile];
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    float x[4] = {__low2float(a), __high2float(a), __low2float(b), __high2float(b)};
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(amax, 448.0f);
    uint32_t codes = 0;
    if (s > 0.f) {
      codes = static_cast<uint32_t>(f32x2_to_e4m3x2(quotient_round_to_odd(x[0], s),
                                                    quotient_round_to_odd(x[1], s))) |
              (static_cast<uint32_t>(f32x2_to_e4m3x2(quotient_round_to_odd(x[2], s),
                                                     quotient_round_to_odd(x[3], s))) << 16);
    }
    *reinterpret_cast<uint32_t*>(rec + tile * 128 + 4 * lane) = codes;
    scales[tile] = s;
  }
  {  // the 64-wide rope tile: 2 elements per lane
    float x0 = __low2float(in.rope), x1 = __high2float(in.rope);
    float amax = fmaxf(fabsf(x0), fabsf(x1));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(amax, 448.0f);
    uint16_t codes = 0;
    if (s > 0.f) codes = f32x2_to_e4m3x2(quotient_round_to_odd(x0, s), quotient_round_to_odd(x1, s));
    *reinterpret_cast<uint16_t*>(rec + 512 + 2 * lane) = codes;
    scales[4] = s;
  }
  if (lane == 0) {
    *reinterpret_cast<uint4*>(rec + kKvScaleOff) =
        make_uint4(__float_as_uint(scales[0]), __float_as_uint(scales[1]),
                   __float_as_uint(scales[2]), __float_as_uint(scales[3]));
  } else if (lane == 1) {
    *reinterpret_cast<uint4*>(rec + kKvScaleOff + 16) = make_uint4(__float_as_uint(scales[4]), 0u, 0u, 0u);
  }
}

}  // namespace dsa
