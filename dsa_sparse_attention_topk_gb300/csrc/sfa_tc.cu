// Sparse Flash Attention on the 5th-generation tensor cores.
//
// "Deep Dive into Sparse Attention and Engineering Optimizations for Efficient Inference
// in Kimi K3.1 Pro", section 1 (attention only over the selected positions) and "Adapting
// and Optimizing Kimi K3.1 Pro for Long-Sequence Inference", section 2 (the cache entries
// named by the indexer's indices are gathered directly); "Kimi K3.1 Pro Inference
// Acceleration: Day0 Optimization on Heterogeneous AI Hardware", sections "FP8 KVCache
// with Per-Token-Head-Tile Quantization for SFA" (FP8 codes with a scale per 128-element
// tile) and "Preserving a Mixed-Precision Path" (BF16 query and attention weighting).
//
// Absorbed MLA decode: each selected position j gives one dequantised latent row kv[j]
// (576 wide); it is the key and kv[j][0:512] is the value.
//
// One CTA handles one query row, one contiguous share ("split") of its selected entries
// and one half of the 512 value columns, for all heads at once (M = 128 rows of the MMAs;
// rows >= h_s are zero).  The two CTAs of a (row, split) compute the same logits and the
// same weights (the same instructions on the same data), so each finishes its own half of
// the output with no exchange.  Halving the output accumulator leaves tensor memory for
// the query's first 384 dims, which then feed Q K^T straight from TMEM; only the last 192
// dims are read from shared memory, and the room this frees holds four KV buffers, so the
// gather runs up to three tiles ahead of the tensor cores.
//
// Twenty-three warps, each role in its own warps:
//   warps 0, 1    Q K^T of the even / odd tiles (32 entries x 576) into their own S buffer
//                 (24 K-steps with the query in TMEM, 12 with it in shared memory); warp 0
//                 also loads the shared-memory part of Q (TMA).
//   warps 4-11    S -> P for entries 0..15 (warps 4-7) and 16..31 (warps 8-11) of a tile,
//                 one head per thread (TMEM lane quadrant = warp mod 4): the two warps of
//                 a quadrant share each tile's maximum through shared memory, keep a
//                 lazily updated running max (the accumulator is rescaled only when the
//                 max grows by more than 2^8) and write P as bf16 over their own S columns.
//                 At the start they store the query's TMEM part.
//   warp 22       P V (A = P from TMEM, B = the tile's value half from shared memory); it
//                 alone waits for each product and publishes how many have completed, which
//                 the S -> P warps read only when they must rescale O.
//   warps 2, 3, 12-21  gather: index -> page -> record, 16-byte loads of E4M3 codes, times
//                 the tile scale, bf16 into the 128-byte-swizzled operand tile (four
//                 buffers; the next tile's codes are converted in registers before its
//                 buffer is free).  Invalid entries (-1, or past the sequence) become zero
//                 rows.  Twelve warps, three on each SM sub-partition, so that the
//                 conversion's instruction stream is spread evenly.
// TMEM (512 columns): O (128 x 256 fp32) in 0..255, S buffers in 256..287 / 288..319 (P
// over columns 0..7 and 16..23 of its buffer), Q dims 0..383 (bf16 pairs) in 320..511.
// Several splits of a row write partial outputs (each normalised by its own sum, bf16)
// with their running max and sums to the workspace; a small kernel merges them.

#include <algorithm>
#include <cfloat>
#include <cuda.h>
#include <mutex>

#include "dsa_common.cuh"
#include "dsa_launch.h"
#include "tc_utils.cuh"

namespace dsa {
namespace {

constexpr int kTok = 32;                       // selected entries per tile
constexpr int kHalfV = kVDim / 2;              // value columns per CTA
constexpr int kWarpQK = 0;                     // warps 0, 1: Q K^T of the even / odd tiles (0: the Q load)
constexpr int kWarpSoft0 = 4;                  // warps 4..11: S -> P
constexpr int kWarpPV = 22;                    // warp 22: P V
constexpr int kGatherWarps = 12;               // warps 2, 3 and 12..21
constexpr int kThreads = 32 * 23;
constexpr int kNumKv = 4;                      // KV buffers (tile j uses buffer j mod 4)
constexpr int kQTmemSteps = 24;                // K-steps of Q K^T with Q in TMEM (dims 0..383)
constexpr int kQBlock = 128 * 128;             // one 64-column K-block of Q: 128 rows x 128 B
constexpr int kQSmemBlocks = 3;                // dims 384..575 in shared memory
constexpr int kQBytes = kQSmemBlocks * kQBlock;  // 49152
constexpr int kKvBlock = kTok * 128;           // one 64-column K-block of a tile: 4096 B
constexpr int kKvBytes = 9 * kKvBlock;         // 36864
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 320;
constexpr int kChunks = kLatent / 16;          // 16-byte code chunks per entry (36)
constexpr int kMaxSplit = 16;
constexpr float kRescaleLog2 = 8.0f;           // lazy max update threshold (factor 256)

struct Ctl {
  uint64_t q_full;             // the shared-memory part of Q has landed (TMA)
  uint64_t q_tmem;             // the TMEM part of Q is stored (8 softmax warps)
  uint64_t kv_full[kNumKv];    // gather -> everyone: tile in buffer k
  uint64_t kv_empty[kNumKv];   // the P V product of the tile in buffer k has completed
  uint64_t s_full[2];          // S of the tile in S buffer b is ready
  uint64_t s_free[2];          // the P in S buffer b has been consumed by its P V product
  uint64_t p_full[2];          // P of the tile in S buffer b is in TMEM and O is rescaled (8 arrivals)
  uint64_t p_done;             // the P V product of the tile has completed (the P V warp waits)
  uint32_t tmem_base;
  int abort;
  int pv_count;                // P V products known complete (written by the P V warp)
  uint8_t valid[kNumKv][kTok]; // per KV buffer: selected entry t of the tile is a real cache row
};

constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKv = kQBytes;
constexpr uint32_t kOffCtl = kOffKv + kNumKv * kKvBytes;
constexpr uint32_t kCtlBytes = 512;
constexpr uint32_t kOffMx = kOffCtl + kCtlBytes;  // [2 tile parities][2 halves][128] tile maxima
constexpr uint32_t kMxBytes = 2 * 2 * 128 * 4;
// At the end the idle KV buffers hold the staged output rows and the final (max, sums).
constexpr int kStagePitch = kHalfV * 2 + 16;   // staged bf16 output row (padded against bank conflicts)
constexpr uint32_t kOffStage = kOffKv;
constexpr uint32_t kOffFin = kOffKv + 2 * kKvBytes;
static_assert(128 * kStagePitch <= 2 * kKvBytes, "the output rows are staged in KV buffers 0 and 1");
// The dynamic shared memory starts 1024-byte aligned (it follows the block's reserved
// 1 KB); the kernel checks this and refuses to run otherwise.
constexpr uint32_t kSmemBytes = kOffMx + kMxBytes;
static_assert(sizeof(Ctl) <= kCtlBytes, "control block");
static_assert(kSmemBytes <= 232448, "shared memory");

__host__ __device__ inline int split_count(int n_q, int topk, int n_sm) {
  const int tiles = (topk + kTok - 1) / kTok;
  int s = n_sm / (2 * (n_q > 0 ? n_q : 1));
  s = s < 1 ? 1 : s;
  s = s > kMaxSplit ? kMaxSplit : s;
  return s > tiles ? tiles : s;
}

int sm_count() {
  DevInfo di;
  const char* why = nullptr;
  return device_info(&di, &why) ? di.n_sm : 152;
}

struct SfaPlan {
  int nsplit, tiles_total;
  __nv_bfloat16* ws_o;  // [n_q][nsplit][h_s][512] partial outputs, each normalised by its own sum l
  float* ws_ml;         // [n_q][nsplit][h_s][4] running max (log2 domain), rounded and exact sums
};

// 2^x with the hardware approximation (relative error ~2^-22; subnormal results flush to
// zero, which is below what the bf16 weights can hold anyway); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// D (+)= A * B with bf16 operands and fp32 accumulation, issued by one elected lane of a
// converged warp (every lane executes the instruction stream; only the elected one
// issues: a converged warp issues MMAs at a steadier rate than a single active lane).
// The _ts form takes A (M = 128 rows, K = 16 bf16 per row as 8 packed columns) from TMEM.
__device__ __forceinline__ void mma_bf16_ts_el(uint32_t d, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               bool accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
      :: "r"(d), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(static_cast<uint32_t>(accumulate))
      : "memory");
}
__device__ __forceinline__ void mma_bf16_ss_el(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               bool accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
      :: "r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(static_cast<uint32_t>(accumulate))
      : "memory");
}
// tcgen05.commit from the elected lane of a converged warp (the lane that issued the MMAs)
__device__ __forceinline__ void commit_el(uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}"
      :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" :: "r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
// Wait until at least n P V products are known complete (bounded like the mbarrier waits).
__device__ __forceinline__ bool wait_pv_count(const int* cnt, int n, volatile int* abort, unsigned* status) {
  if (ld_acquire(cnt) >= n) return true;
  const uint64_t t0 = tc::global_ns();
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire(cnt) >= n) return true;
    if ((it & 255u) == 255u) {
      if (*abort) return false;
      if (tc::global_ns() - t0 > tc::kWaitLimitNs) {
        *abort = 1;
        flag(status, DSA_STATUS_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
         "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
         "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
         "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
sfa_tc_kernel(const __grid_constant__ CUtensorMap qmap, SfaArgs a, SfaPlan pl) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* s_q = smem + kOffQ;
  uint8_t* s_kv = smem + kOffKv;
  Ctl& ctl = *reinterpret_cast<Ctl*>(smem + kOffCtl);
  float* s_mx = reinterpret_cast<float*>(smem + kOffMx);  // [2][2][128]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x >> 1, half = blockIdx.x & 1, t = blockIdx.y;
  const int tile0 = split * pl.tiles_total / pl.nsplit;
  const int nt = (split + 1) * pl.tiles_total / pl.nsplit - tile0;
  // every swizzled operand tile needs 1024-byte alignment (uniform over the block)
  if (smem_u32(smem) & 1023u) {
    if (tid == 0) flag(a.status, DSA_STATUS_INTERNAL);
    return;
  }

  if (tid == 0) {
    ctl.abort = 0;
    tc::mbar_init(&ctl.q_full, 1);
    tc::mbar_init(&ctl.q_tmem, 8);
    for (int k = 0; k < kNumKv; ++k) {
      tc::mbar_init(&ctl.kv_full[k], kGatherWarps);
      tc::mbar_init(&ctl.kv_empty[k], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&ctl.s_full[b], 1);
      tc::mbar_init(&ctl.s_free[b], 1);
    }
    tc::mbar_init(&ctl.p_full[0], 8);
    tc::mbar_init(&ctl.p_full[1], 8);
    tc::mbar_init(&ctl.p_done, 1);
    ctl.pv_count = 0;
    tc::mbar_fence_init();
  }
  if (warp == 0) tc::tmem_alloc(&ctl.tmem_base, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort = &ctl.abort;

  pdl_launch_dependents();
  pdl_wait();  // nothing global is touched before the previous kernel on the stream is done
  const int seq = a.q_seq[t];
  const bool seq_ok = seq >= 0 && seq < a.n_seq;
  const int L = seq_ok ? a.seq_lens[seq] : 0;
  const int32_t* ptab = a.page_table + static_cast<size_t>(seq_ok ? seq : 0) * a.max_pages;
  const int32_t* idx = a.idx + static_cast<size_t>(t) * a.topk;
  if (tid == 0 && !seq_ok && split == 0 && half == 0) flag(a.status, DSA_STATUS_BAD_SEQ);

  if (warp == kWarpQK || warp == kWarpQK + 1) {
    // ---------------- Q K^T issuers ----------------
    // warp kWarpQK + b issues the tiles j = b (mod 2) from lane 0 into S buffer b; they sit
    // in KV buffers b and b + 2 in turn, so the loop takes them two at a time and every
    // operand address stays fixed.  Two issuing warps, because one thread issues an MMA
    // only every ~45 cycles.
    const int b = warp - kWarpQK;
    if (b == 0 && lane == 0) {
      tc::prefetch_tmap(&qmap);
      tc::mbar_arrive_expect_tx(&ctl.q_full, kQBytes);
      for (int kb = 0; kb < kQSmemBlocks; ++kb)
        tc::tma_load_3d(s_q + kb * kQBlock, &qmap, kQTmemSteps * 16 + kb * 64, 0, t, &ctl.q_full);
    }
    __syncwarp();
    const uint32_t id_qk = tc::idesc_bf16(kTok, false, false);
    tc::mbar_wait(&ctl.q_full, 0, abort, a.status);
    tc::mbar_wait(&ctl.q_tmem, 0, abort, a.status);
    // descriptors advance by adding (byte offset >> 4) to the start-address field
    const uint64_t qd = tc::desc_kmajor_sw128(smem_u32(s_q));
    const uint32_t d = tmem + kColS + kTok * b;
    auto qk = [&](int j, uint64_t kd) {
      tc::mbar_wait(&ctl.kv_full[j & 3], (j >> 2) & 1, abort, a.status);
      tc::mbar_wait(&ctl.s_free[b], ((j >> 1) & 1) ^ 1, abort, a.status);
      __syncwarp();
      tc::fence_after_sync();
#pragma unroll
      for (int st = 0; st < kQTmemSteps; ++st)  // dims 16 st .. : Q from TMEM
        mma_bf16_ts_el(d, tmem + kColQ + 8 * st, kd + ((st >> 2) * (kKvBlock >> 4) + 2 * (st & 3)), id_qk, st > 0);
#pragma unroll
      for (int st = kQTmemSteps; st < 36; ++st) {  // dims 384.. : Q from shared memory
        const int qs = st - kQTmemSteps;
        mma_bf16_ss_el(d, qd + ((qs >> 2) * (kQBlock >> 4) + 2 * (qs & 3)),
                       kd + ((st >> 2) * (kKvBlock >> 4) + 2 * (st & 3)), id_qk, true);
      }
      commit_el(&ctl.s_full[b]);
    };
    const uint64_t kd0 = tc::desc_kmajor_sw128(smem_u32(s_kv + b * kKvBytes));
    const uint64_t kd1 = tc::desc_kmajor_sw128(smem_u32(s_kv + (b + 2) * kKvBytes));
    for (int j = b; j < nt; j += 4) {
      qk(j, kd0);
      if (j + 2 < nt) qk(j + 2, kd1);
    }
    __syncwarp();
  } else if (warp >= kWarpSoft0 && warp < kWarpSoft0 + 8) {
    // ---------------- S -> P (warps 4..11) ----------------
    const int quarter = warp & 3;
    const int hv = (warp - kWarpSoft0) >> 2;  // entries 16 hv .. 16 hv + 15 of every tile
    const int m = quarter * 32 + lane;        // head row
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    // the query's first 384 dims into TMEM (dims 192 hv .. +191 of head m, bf16 pairs)
    {
      uint32_t r[32];
#pragma unroll
      for (int h3 = 0; h3 < 3; ++h3) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                          (static_cast<size_t>(t) * a.h_s + m) * kLatent +
                                                          192 * hv + 64 * h3);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (m < a.h_s) v = __ldg(src + i);
          r[4 * i] = v.x; r[4 * i + 1] = v.y; r[4 * i + 2] = v.z; r[4 * i + 3] = v.w;
        }
        tmem_st32(tmem + lane_base + kColQ + 96 * hv + 32 * h3, r);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&ctl.q_tmem);
    }
    const float c2 = a.sm_scale * 1.4426950408889634f;  // logits in log2 units
    // l sums the bf16-rounded weights that the P V product uses (it normalises O);
    // lx sums the unrounded weights (it gives the log-sum-exp)
    float m_ref = -INFINITY, l = 0.f, lx = 0.f;
    const uint32_t bar_pair = 1 + quarter;            // named barrier of the quadrant's two warps
    for (int j = 0; j < nt; ++j) {
      const int b = j & 1, kb = j & 3;
      // the gather warps flag the tile's real entries before they release the buffer
      tc::mbar_wait(&ctl.kv_full[kb], (j >> 2) & 1, abort, a.status);
      const uint32_t mask = __ballot_sync(0xffffffffu, lane < 16 && ctl.valid[kb][16 * hv + (lane & 15)] != 0);
      tc::mbar_wait(&ctl.s_full[b], (j >> 1) & 1, abort, a.status);
      tc::fence_after_sync();
      const uint32_t sb = tmem + lane_base + kColS + kTok * b + 16 * hv;
      uint32_t sr[16];
      tc::tmem_ld16(sb, sr);
      tc::tmem_wait_ld();
      float x[16];
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        x[i] = ((mask >> i) & 1u) ? __uint_as_float(sr[i]) * c2 : -INFINITY;
        mt = fmaxf(mt, x[i]);
      }
      // the tile's maximum over both halves (slot by tile parity: the partner reads slot
      // j & 1 before it passes the barrier of tile j + 1, after which it is rewritten)
      s_mx[((j & 1) * 2 + hv) * 128 + m] = mt;
      asm volatile("bar.sync %0, 64;" :: "r"(bar_pair) : "memory");
      mt = fmaxf(mt, s_mx[((j & 1) * 2 + (hv ^ 1)) * 128 + m]);
      const bool need = mt > m_ref + kRescaleLog2 || (m_ref == -INFINITY && mt > -INFINITY);
      const float m_new = need ? mt : m_ref;
      const float alpha = need ? fast_exp2(m_ref - m_new) : 1.f;  // 2^-inf = 0
      uint32_t pk[8];
      float lsum = 0.f, lxsum = 0.f;
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const float p0 = (m_new == -INFINITY) ? 0.f : fast_exp2(x[i] - m_new);
        const float p1 = (m_new == -INFINITY) ? 0.f : fast_exp2(x[i + 1] - m_new);
        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
        lsum += __low2float(pb) + __high2float(pb);
        lxsum += p0 + p1;
        pk[i >> 1] = *reinterpret_cast<const uint32_t*>(&pb);
      }
      // P over this warp's own (already read) S columns
      tmem_st8(sb, pk);
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // O is rescaled once the previous tile's P V product has completed
        wait_pv_count(&ctl.pv_count, j, abort, a.status);
        tc::fence_after_sync();
        // this warp's half of O's columns
        for (int c = 128 * hv; c < 128 * hv + 128; c += 16) {
          uint32_t r[16];
          tc::tmem_ld16(tmem + lane_base + kColO + c, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tc::tmem_st16(tmem + lane_base + kColO + c, r);
        }
      }
      tc::tmem_wait_st();
      l = l * alpha + lsum;
      lx = lx * alpha + lxsum;
      m_ref = m_new;
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&ctl.p_full[b]);
    }
    // every product has completed; publish (max, sums) for the output phase
    wait_pv_count(&ctl.pv_count, nt, abort, a.status);
    tc::fence_after_sync();
    float* s_fin = reinterpret_cast<float*>(smem + kOffFin);  // [0]: max; [1 + hv]: l; [3 + hv]: lx
    if (hv == 0) s_fin[m] = m_ref;
    s_fin[(1 + hv) * 128 + m] = l;
    s_fin[(3 + hv) * 128 + m] = lx;
  } else if (warp == kWarpPV) {
    // ---------------- P V (warp 22) ----------------
    // O += P V over each tile's 32 entries (2 K-steps of 16): A = P from S buffer b (entries
    // 0..15 in its columns 0..7, 16..31 in 16..23), B = this CTA's value half of the tile
    // (MN-major: 64-column blocks 4096 bytes apart, 8-entry groups 1024 bytes apart).  This
    // warp is the only waiter of p_done and waits for every product in turn, so its parity
    // never falls behind; the products chain through O, so waiting costs only the gap
    // before the next issue.
    const uint32_t id_pv = tc::idesc_bf16(kHalfV, false, true);
    for (int j = 0; j < nt; ++j) {
      const int b = j & 1, kb = j & 3;
      // (one barrier per S buffer: the S -> P warps reach tile j + 2 only after this
      // product has freed the buffer, so the waiter never falls two phases behind)
      tc::mbar_wait(&ctl.p_full[b], (j >> 1) & 1, abort, a.status);
      __syncwarp();
      tc::fence_after_sync();
      const uint32_t pbase = tmem + kColS + kTok * b;
      const uint32_t vaddr = smem_u32(s_kv + kb * kKvBytes + 4 * half * kKvBlock);
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const uint64_t vd = tc::smem_desc(vaddr + ks * 2048, kKvBlock, 1024, 2);
        mma_bf16_ts_el(tmem + kColO, pbase + 16 * ks, vd, id_pv, j > 0 || ks > 0);
      }
      commit_el(&ctl.s_free[b]);
      commit_el(&ctl.kv_empty[kb]);
      commit_el(&ctl.p_done);
      tc::mbar_wait(&ctl.p_done, j & 1, abort, a.status);
      tc::fence_after_sync();
      __syncwarp();
      if (lane == 0) st_release(&ctl.pv_count, j + 1);
    }
  } else {
    // ---------------- gather + dequantise (warps 2, 3, 12..21) ----------------
    // Thread g owns entry tok = g / 12 of every tile and its 16-byte code chunks
    // c = s, s + 12, s + 24 (s = g % 12): one index -> page -> record lookup per tile, and
    // twelve threads read one record's 576 codes in contiguous 192-byte runs.  The loads
    // run ahead of their use: while tile j is converted, the index entry of tile j + 4, the
    // page of tile j + 3, an L2 prefetch of the records of tile j + 2 and the codes of tile
    // j + 1 are in flight, so no iteration waits on a load it issued itself.
    constexpr int kPer = 3;  // chunks per thread
    static_assert(kTok * 12 == 32 * kGatherWarps && kChunks == 12 * kPer, "twelve threads per entry");
    const int g = (warp < 4 ? warp - 2 : warp - 10) * 32 + lane;  // 0..383
    const int tok = g / 12, s12 = g % 12;
    const bool reporter = s12 == 0;             // one thread per entry reports bad input
    auto ld_s32 = [](const int32_t* ptr) {
      int v;
      asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(ptr));
      return v;
    };
    // index entry of tile jj for this thread's entry (-1: past the row, or nothing selected)
    auto entry = [&](int jj) -> int {
      const int e = (tile0 + jj) * kTok + tok;
      return (jj < nt && e < a.topk) ? ld_s32(idx + e) : -1;
    };
    auto in_range = [&](int p) { return p >= 0 && p < L && p / kPage < a.max_pages; };
    // physical page of position p (-1 when p is out of range)
    auto page_of = [&](int p) -> int { return in_range(p) ? ld_s32(ptab + p / kPage) : -1; };
    uint4 code[kPer];
    float scl[kPer];
    bool live = false;
    // request the codes of the entry at position p on page pg
    auto load_codes = [&](int p, int pg) {
      live = false;
      const uint8_t* rec = nullptr;
      if (p >= 0) {
        if (!in_range(p)) {
          if (reporter) flag(a.status, DSA_STATUS_BAD_INDEX);
        } else if (pg < 0 || pg >= a.num_pages) {
          if (reporter) flag(a.status, DSA_STATUS_BAD_PAGE);
        } else {
          rec = a.kv_cache + (static_cast<int64_t>(pg) * kPage + p % kPage) * kKvTokBytes;
        }
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        code[k] = make_uint4(0u, 0u, 0u, 0u);
        scl[k] = 0.f;
      }
      if (rec) {
        live = true;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int c = s12 + 12 * k;
          asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(code[k].x), "=r"(code[k].y), "=r"(code[k].z), "=r"(code[k].w)
                       : "l"(rec + 16 * c));
          asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];"
                       : "=f"(scl[k]) : "l"(rec + kKvScaleOff + 4 * (c >> 3)));
        }
      }
    };
    // pull the 608-byte record of the entry at position p on page pg towards L2 (five of
    // the entry's twelve threads take one 128-byte line each)
    auto prefetch_record = [&](int p, int pg) {
      if (s12 < 5 && in_range(p) && pg >= 0 && pg < a.num_pages) {
        const uint8_t* rec = a.kv_cache + (static_cast<int64_t>(pg) * kPage + p % kPage) * kKvTokBytes;
        asm volatile("prefetch.global.L2 [%0];" :: "l"(rec + min(128 * s12, kKvTokBytes - 1)));
      }
    };
    // warm L2 with this split's index entries and the sequence's page-table row (one
    // 128-byte line per thread), so that the first lookups do not each pay a DRAM access
    {
      const int e_lo = tile0 * kTok, e_hi = min(a.topk, (tile0 + nt) * kTok);
      const int npg = min(a.max_pages, (L + kPage - 1) / kPage);
      for (int e = e_lo + 32 * g; e < e_hi; e += 32 * 32 * kGatherWarps)
        asm volatile("prefetch.global.L2 [%0];" :: "l"(idx + e));
      for (int i = 32 * g; i < npg; i += 32 * 32 * kGatherWarps)
        asm volatile("prefetch.global.L2 [%0];" :: "l"(ptab + i));
    }
    // prologue: index entries of tiles 0..3, pages of 0..2, the record of 1 towards L2 and
    // the codes of tile 0
    int p1 = entry(0), p2 = entry(1), p3 = entry(2), p4 = entry(3);
    int pg1 = page_of(p1), pg2 = page_of(p2), pg3 = page_of(p3);
    prefetch_record(p2, pg2);
    load_codes(p1, pg1);
    p1 = p2; pg1 = pg2; p2 = p3; pg2 = pg3; p3 = p4;
    for (int j = 0; j < nt; ++j) {
      const int kb = j & 3;
      uint8_t* kv = s_kv + kb * kKvBytes;
      // requests for the tiles ahead: the index of j + 4, the page of j + 3 and the record of
      // j + 2 (towards L2) now, the codes of j + 1 once this tile's have left their registers
      const int p4n = entry(j + 4);
      const int pg3n = page_of(p3);
      prefetch_record(p2, pg2);
      // this tile's codes -> bf16 in registers
      uint4 o0s[kPer], o1s[kPer];
      const bool live_j = live;
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const uint32_t w[4] = {code[k].x, code[k].y, code[k].z, code[k].w};
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float f[4];
          e4m3x4_to_f32(w[q], f);
          o[2 * q] = pack_bf16(f[0] * scl[k], f[1] * scl[k]);
          o[2 * q + 1] = pack_bf16(f[2] * scl[k], f[3] * scl[k]);
        }
        o0s[k] = make_uint4(o[0], o[1], o[2], o[3]);
        o1s[k] = make_uint4(o[4], o[5], o[6], o[7]);
        // pin the converted words here: left to itself the compiler moves the conversion
        // behind the wait below, where it delays the tile by its whole length
        asm volatile("" : "+r"(o0s[k].x), "+r"(o0s[k].y), "+r"(o0s[k].z), "+r"(o0s[k].w),
                          "+r"(o1s[k].x), "+r"(o1s[k].y), "+r"(o1s[k].z), "+r"(o1s[k].w));
      }
      load_codes(p1, pg1);
      p1 = p2; pg1 = pg2; p2 = p3; pg2 = pg3n; p3 = p4n;
      tc::mbar_wait(&ctl.kv_empty[kb], ((j >> 2) & 1) ^ 1, abort, a.status);
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int c = s12 + 12 * k;
        const int kblk = c >> 2, cc = (c & 3) * 2;
        uint8_t* row = kv + kblk * kKvBlock + tok * 128;
        *reinterpret_cast<uint4*>(row + ((cc ^ (tok & 7)) << 4)) = o0s[k];
        *reinterpret_cast<uint4*>(row + (((cc + 1) ^ (tok & 7)) << 4)) = o1s[k];
      }
      if (reporter) ctl.valid[kb][tok] = live_j ? 1 : 0;
      tc::fence_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&ctl.kv_full[kb]);
    }
  }
  // ---- the output rows, normalised, as bf16: to the output (one split) or to the
  // workspace (several splits; merged by sfa_combine_kernel).  Warp w reads its lane
  // quadrant (w mod 4), columns 64 (w / 4) .. +64, and stages them in the idle KV buffers;
  // then every warp writes whole rows, 512 contiguous bytes per instruction. ----
  tc::fence_before_sync();
  __syncthreads();  // the S -> P warps have seen the last product complete and published (m, l, lx)
  tc::fence_after_sync();
  uint8_t* s_stage = smem + kOffStage;
  {
    const float* s_fin = reinterpret_cast<const float*>(smem + kOffFin);
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float l = s_fin[128 + m] + s_fin[256 + m];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint8_t* row = s_stage + m * kStagePitch;
    const int cbeg = 64 * (warp >> 2);
#pragma unroll
    for (int c = cbeg; c < cbeg + 64 && warp < 16; c += 32) {
      uint32_t r[32];
      if (nt > 0) {
        tc::tmem_ld32(tmem + lane_base + kColO + c, r);
        tc::tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = 0u;
      }
#pragma unroll
      for (int i = 0; i < 32; i += 8)
        *reinterpret_cast<uint4*>(row + 2 * (c + i)) =
            make_uint4(pack_bf16(__uint_as_float(r[i]) * inv, __uint_as_float(r[i + 1]) * inv),
                       pack_bf16(__uint_as_float(r[i + 2]) * inv, __uint_as_float(r[i + 3]) * inv),
                       pack_bf16(__uint_as_float(r[i + 4]) * inv, __uint_as_float(r[i + 5]) * inv),
                       pack_bf16(__uint_as_float(r[i + 6]) * inv, __uint_as_float(r[i + 7]) * inv));
    }
    if (half == 0 && m < a.h_s && warp >= kWarpSoft0 && warp < kWarpSoft0 + 4) {
      const float m_ref = s_fin[m], lx = s_fin[384 + m] + s_fin[512 + m];
      const size_t slot = (static_cast<size_t>(t) * pl.nsplit + split) * a.h_s + m;
      if (pl.nsplit == 1) {
        if (a.out_lse)
          a.out_lse[static_cast<size_t>(t) * a.h_s + m] = lx > 0.f ? (m_ref + log2f(lx)) * 0.6931471805599453f : -INFINITY;
      } else {
        *reinterpret_cast<float4*>(pl.ws_ml + 4 * slot) = make_float4(m_ref, l, lx, 0.f);
      }
    }
  }
  __syncthreads();  // every staged row is complete
  {
    // row h: 32 pieces of 16 bytes; warp w writes rows w, w + 23, ..
    const int piece = tid & 31;
    for (int h = tid >> 5; h < a.h_s; h += kThreads / 32) {
      __nv_bfloat16* dst = pl.nsplit == 1
                               ? static_cast<__nv_bfloat16*>(a.out) + (static_cast<size_t>(t) * a.h_s + h) * kVDim
                               : pl.ws_o + ((static_cast<size_t>(t) * pl.nsplit + split) * a.h_s + h) * kVDim;
      *reinterpret_cast<uint4*>(dst + kHalfV * half + 8 * piece) =
          *reinterpret_cast<const uint4*>(s_stage + h * kStagePitch + 16 * piece);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// Merge the splits of each (row, head).  Split s holds O_s / l_s with running max m_s; with
// M = max_s m_s and c_s = 2^(m_s - M) l_s the output is sum_s c_s (O_s / l_s) / sum_s c_s.
// 64 threads per (row, head), 8 value dims each, four heads per block.  The splits are
// taken four at a time with all their loads issued before any is used (the merge is bound
// by the latency of those loads, not by bandwidth); a later group whose max is larger
// rescales what has been summed so far.
constexpr int kCombineHeads = 4;
constexpr int kCombineBatch = 4;
__global__ void __launch_bounds__(64 * kCombineHeads)
sfa_combine_kernel(SfaArgs a, SfaPlan pl) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x;
  const int h = blockIdx.y * kCombineHeads + static_cast<int>(threadIdx.x >> 6);
  if (h >= a.h_s) return;
  const int d = 8 * static_cast<int>(threadIdx.x & 63);
  const int ns = pl.nsplit;
  const size_t slot0 = static_cast<size_t>(t) * ns * a.h_s + h;  // split s: slot0 + s h_s
  float M = -INFINITY, csum = 0.f, wsum_x = 0.f;
  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.f;
  for (int s0 = 0; s0 < ns; s0 += kCombineBatch) {
    float4 ml[kCombineBatch];
    uint4 v[kCombineBatch];
#pragma unroll
    for (int i = 0; i < kCombineBatch; ++i) {
      if (s0 + i < ns) {
        const size_t slot = slot0 + static_cast<size_t>(s0 + i) * a.h_s;
        ml[i] = *reinterpret_cast<const float4*>(pl.ws_ml + 4 * slot);
        v[i] = *reinterpret_cast<const uint4*>(pl.ws_o + slot * kVDim + d);
      } else {
        ml[i] = make_float4(-INFINITY, 0.f, 0.f, 0.f);
        v[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float Mn = M;
#pragma unroll
    for (int i = 0; i < kCombineBatch; ++i) Mn = fmaxf(Mn, ml[i].x);
    if (Mn != M) {  // (the first group: everything so far is zero)
      const float r = M == -INFINITY ? 0.f : exp2f(M - Mn);
      csum *= r;
      wsum_x *= r;
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] *= r;
      M = Mn;
    }
#pragma unroll
    for (int i = 0; i < kCombineBatch; ++i) {
      const float wgt = (ml[i].x == -INFINITY) ? 0.f : exp2f(ml[i].x - M);
      const float c = wgt * ml[i].y;
      csum += c;
      wsum_x += wgt * ml[i].z;
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
        acc[2 * k] += c * __low2float(p);
        acc[2 * k + 1] += c * __high2float(p);
      }
    }
  }
  const float inv = csum > 0.f ? 1.f / csum : 0.f;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (static_cast<size_t>(t) * a.h_s + h) * kVDim;
  *reinterpret_cast<uint4*>(out + d) =
      make_uint4(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv),
                 pack_bf16(acc[4] * inv, acc[5] * inv), pack_bf16(acc[6] * inv, acc[7] * inv));
  if (a.out_lse && d == 0)
    a.out_lse[static_cast<size_t>(t) * a.h_s + h] =
        wsum_x > 0.f ? (M + log2f(wsum_x)) * 0.6931471805599453f : -INFINITY;
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

size_t ws_o_bytes(int n_q, int h_s, int ns) {
  return (static_cast<size_t>(n_q) * ns * h_s * kVDim * sizeof(__nv_bfloat16) + 255) / 256 * 256;
}

}  // namespace

size_t sfa_workspace_bytes(int n_q, int h_s, int topk) {
  const int ns = split_count(n_q, topk, sm_count());
  if (ns <= 1) return 0;
  return ws_o_bytes(n_q, h_s, ns) + static_cast<size_t>(n_q) * ns * h_s * 4 * sizeof(float);
}

cudaError_t launch_sfa(const SfaArgs& a, cudaStream_t s, const char** err) {
  if (a.n_q == 0) return cudaSuccess;
  SfaPlan pl{};
  pl.nsplit = split_count(a.n_q, a.topk, sm_count());
  pl.tiles_total = (a.topk + kTok - 1) / kTok;
  if (pl.nsplit > 1) {
    pl.ws_o = static_cast<__nv_bfloat16*>(a.workspace);
    pl.ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + ws_o_bytes(a.n_q, a.h_s, pl.nsplit));
  }
  EncodeFn enc = encode_fn();
  if (!enc) {
    *err = "sparse_attn: cuTensorMapEncodeTiled is not available";
    return cudaErrorNotSupported;
  }
  CUtensorMap qmap;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kLatent), static_cast<cuuint64_t>(a.h_s),
                              static_cast<cuuint64_t>(a.n_q)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kLatent) * 2,
                                 static_cast<cuuint64_t>(kLatent) * 2 * static_cast<cuuint64_t>(a.h_s)};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
    *err = "sparse_attn: tensor map encoding failed";
    return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(sfa_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  e = launch_pdl(sfa_tc_kernel, dim3(2 * pl.nsplit, a.n_q), dim3(kThreads), kSmemBytes, s, 1, qmap, a, pl);
  if (e != cudaSuccess || pl.nsplit == 1) return e;
  return launch_pdl(sfa_combine_kernel, dim3(a.n_q, (a.h_s + kCombineHeads - 1) / kCombineHeads),
                    dim3(64 * kCombineHeads), 0, s, 1, a, pl);
}

// ---- scratch for callers that cannot allocate ----------------------------------------
// Some callers of this library have no way to allocate device memory for the split-merge
// workspace: code running under a caching allocator they may not bypass, inside a
// framework that owns every allocation, or on a path where an allocation call would
// synchronise the device.  For them the partial outputs go to this fixed array instead.
// It lives for as long as the library is loaded on a device, is shared by every call on
// that device, and keeps the last call's contents (nothing in it needs to start at zero:
// every slot is written before it is read).  Two calls whose kernels overlap on the GPU
// would race on it.
static __device__ __align__(256) unsigned char g_sfa_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];

cudaError_t launch_sfa_noalloc(const SfaArgs& a_in, cudaStream_t s, const char** err) {
  const size_t need = sfa_workspace_bytes(a_in.n_q, a_in.h_s, a_in.topk);
  if (need > sizeof(g_sfa_noalloc_scratch)) {
    *err = "sparse_attn_noalloc: these sizes need more scratch than DSA_NOALLOC_SCRATCH_BYTES";
    return cudaErrorInvalidValue;
  }
  // The host-side name of the array is only a stand-in; the device address comes from
  // cudaGetSymbolAddress, looked up once per device with that device current.
  static std::mutex mu;
  static void* ptrs[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) {
    *err = "sparse_attn_noalloc: device ordinal out of range";
    return cudaErrorInvalidDevice;
  }
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
      e = cudaGetSymbolAddress(&ptrs[dev], g_sfa_noalloc_scratch);
      if (e != cudaSuccess) {
        ptrs[dev] = nullptr;
        return e;
      }
    }
    ptr = ptrs[dev];
  }
  SfaArgs a = a_in;
  a.workspace = ptr;
  a.workspace_bytes = sizeof(g_sfa_noalloc_scratch);
  return launch_sfa(a, s, err);
}

}  // namespace dsa
