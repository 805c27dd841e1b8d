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
// One CTA handles one query row and one contiguous share ("split") of its selected
// entries, for all heads at once (M = 128 rows of the MMAs; rows >= h_s are zero).
// Sixteen warps, each role in its own warps so that no role's latency sits in another's
// loop:
//   warps 0, 1  Q K^T of the even and the odd tiles: Q (bf16, 128 x 576, resident, loaded
//               once by TMA) times a gathered tile (32 entries x 576) into one of two S
//               buffers in TMEM, so the next tile's QK^T runs while the softmax works on this
//               one.  Two issuing warps, because a single thread issues an MMA only every
//               ~55 cycles while the operand reads of one take ~40.
//   warps 4-7   S -> P, one head per thread: online softmax in the exp2 domain with a
//               lazily updated running max (the accumulator is rescaled only when the max
//               grows by more than 2^8), P written to shared memory as bf16.
//   warps 8-11  the tail rounds, added into register accumulators (rescaled with the max
//               that the S -> P warps publish per tile).
//   lane 0 of warp 4 also issues every P V once the tile's P is stored: O[:, 0:448] into
//               its TMEM accumulator, and O[:, 448:512] in two 32-column rounds through the
//               tile's S buffer (free once its S was read).  The first round goes ahead of
//               the large products, so the tail warps read it while those run; the second
//               is issued at the start of the next tile, so the softmax never waits for it.
//   warps 2, 3, 12-15  gather: index -> page -> record, 16-byte loads of E4M3 codes,
//               multiply by the tile scale, bf16 into the 128-byte-swizzled operand tile
//               (double buffered; the next tile's codes are loaded and converted in
//               registers before its buffer is free).  Invalid entries (-1, or past the
//               sequence) become zero rows.
// TMEM (512 columns): O[:, 0:448] in columns 0..447, S buffers in 448..479 (even tiles)
// and 480..511 (odd tiles).  At N = 32 an MMA costs ~40 cycles of the SM's operand reads
// whatever issues it (a 4 KB Q slice and a 1 KB tile slice from shared memory), so QK^T's
// 36 K-steps are the largest cost of a tile.  With two KV buffers next to the resident Q,
// a buffer is refilled only after its tile's P V products, so the chain gather -> Q K^T ->
// softmax -> P V -> tail rounds, once per two tiles, sets the pace (~4400 cycles a tile).
// Several splits of a row write their partial outputs (each normalised by its own sum,
// bf16) with their running max and sums to the workspace; a small kernel merges them
// (log-sum-exp weights).  (Merging inside
// a cluster of the row's splits, through distributed shared memory or through L2, measured
// slower: the split-merge kernel runs spread over the whole GPU.)

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
constexpr int kWarpQK = 0;                     // warps 0, 1: Q K^T of the even / odd tiles (0: the Q load)
constexpr int kWarpSoft0 = 4;                  // warps 4..7: S -> P, one TMEM lane quadrant each; warp 4 issues P V
constexpr int kWarpTail0 = 8;                  // warps 8..11: tail rounds, one quadrant each
constexpr int kGatherWarps = 6;                // warps 2, 3 and 12..15
constexpr int kThreads = 512;
constexpr int kQBlock = 128 * 128;             // one 64-column K-block of Q: 128 rows x 128 B
constexpr int kQBytes = 9 * kQBlock;           // 147456
constexpr int kKvBlock = kTok * 128;           // one 64-column K-block of a tile: 4096 B
constexpr int kKvBytes = 9 * kKvBlock;         // 36864
constexpr int kPBytes = 128 * kTok * 2;        // 8192
constexpr uint32_t kColS = 448;                // S buffers (tile j: kColS + 32 (j & 1)), tail rounds
constexpr int kVLeft = 448;                    // output columns accumulated in TMEM
constexpr int kVTail = 64;                     // output columns accumulated in registers
constexpr int kChunks = kLatent / 16;          // 16-byte code chunks per entry (36)
constexpr int kSplitTarget = 148;              // CTAs the split count aims for
constexpr int kMaxSplit = 16;
constexpr float kRescaleLog2 = 8.0f;           // lazy max update threshold (factor 256)

// Every barrier waited on by parity has waiters that cannot fall two phases behind: each
// next phase needs something the waiters do after their wait.
struct Ctl {
  uint64_t q_full;
  uint64_t kv_full[2];     // gather -> everyone: tile in buffer b
  uint64_t kv_empty[2];    // QK^T and the P V products of the tile are done with buffer b
  uint64_t s_full[2];      // S of the tile in S buffer b is ready
  uint64_t s_free[2];      // S buffer b is free again (its tail rounds have been read)
  uint64_t p_full;         // P of the tile is in shared memory
  uint64_t p_free;         // every P V product of the tile has completed
  uint64_t m_ready[2];     // the running max of the tile in S buffer b is in s_m[b]
  uint64_t tail_full[2];   // a tail round is in S buffer b (two phases per tile)
  uint64_t tail_empty;     // the first tail round has been read
  uint32_t tmem_base;
  int abort;
  uint8_t valid[2][kTok];  // per KV buffer: selected entry t of the tile is a real cache row
};

constexpr uint32_t kOffQ = 0;
constexpr int kStagePitch = kVDim * 2 + 16;    // staged bf16 output row (padded against bank conflicts)
static_assert(128 * kStagePitch <= kQBytes, "the output rows are staged in the Q buffer");
constexpr uint32_t kOffKv = kQBytes;
constexpr uint32_t kOffP = kOffKv + 2 * kKvBytes;
constexpr uint32_t kOffCtl = kOffP + kPBytes;
constexpr uint32_t kCtlBytes = 256;
constexpr uint32_t kOffM = kOffCtl + kCtlBytes;  // running max of each head, per tile parity
constexpr uint32_t kMBytes = 2 * 128 * 4;
constexpr uint32_t kSmemBytes = kOffM + kMBytes + 1024;  // + slack for the 1024-byte alignment
static_assert(sizeof(Ctl) <= kCtlBytes, "control block");

__host__ __device__ inline int split_count(int n_q, int topk) {
  const int tiles = (topk + kTok - 1) / kTok;
  int s = kSplitTarget / (n_q > 0 ? n_q : 1);
  s = s < 1 ? 1 : s;
  s = s > kMaxSplit ? kMaxSplit : s;
  return s > tiles ? tiles : s;
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

__global__ void __launch_bounds__(kThreads, 1)
sfa_tc_kernel(const __grid_constant__ CUtensorMap qmap, SfaArgs a, SfaPlan pl) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* s_q = smem + kOffQ;
  uint8_t* s_kv = smem + kOffKv;
  uint8_t* s_p = smem + kOffP;
  Ctl& ctl = *reinterpret_cast<Ctl*>(smem + kOffCtl);
  float* s_m = reinterpret_cast<float*>(smem + kOffM);  // [2][128]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, t = blockIdx.y;
  const int tile0 = split * pl.tiles_total / pl.nsplit;
  const int nt = (split + 1) * pl.tiles_total / pl.nsplit - tile0;

  if (tid == 0) {
    ctl.abort = 0;
    tc::mbar_init(&ctl.q_full, 1);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&ctl.kv_full[b], kGatherWarps);
      tc::mbar_init(&ctl.kv_empty[b], 2);
      tc::mbar_init(&ctl.s_full[b], 1);
      tc::mbar_init(&ctl.s_free[b], 4);
      tc::mbar_init(&ctl.tail_full[b], 1);
    }
    tc::mbar_init(&ctl.p_full, 4);
    tc::mbar_init(&ctl.p_free, 1);
    tc::mbar_init(&ctl.m_ready[0], 4);
    tc::mbar_init(&ctl.m_ready[1], 4);
    tc::mbar_init(&ctl.tail_empty, 4);
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
  if (tid == 0 && !seq_ok && split == 0) flag(a.status, DSA_STATUS_BAD_SEQ);

  // P V of tile j, issued by one thread: O[:, 0:448] into the TMEM accumulator, and
  // O[:, 448:512] in two 32-column rounds through S buffer j & 1 (its S has been read) that
  // the tail warps add into registers.  The second round waits until the tail warps have
  // read the first, so its issue is deferred to the start of the next tile (pv_second_round),
  // and the issuing thread goes on with the softmax meanwhile.
  const uint32_t id_v0 = tc::idesc_bf16(256, false, true);
  const uint32_t id_v1 = tc::idesc_bf16(192, false, true);
  const uint32_t id_vt = tc::idesc_bf16(kTok, false, true);
  auto pv_desc = [&](int j, int ks, uint64_t& pd, uint64_t& vd) {
    pd = tc::smem_desc(smem_u32(s_p + ks * 256), 128, 512, 0);
    vd = tc::smem_desc(smem_u32(s_kv + (j & 1) * kKvBytes + ks * 2048), kKvBlock, 1024, 2);  // 16 entries = two 8-row groups
  };
  auto pv_main = [&](int j) {
    const int b = j & 1;
    tc::mbar_wait(&ctl.p_full, j & 1, abort, a.status);  // every S -> P warp has stored its rows
    tc::fence_after_sync();
    // the first tail round goes first: the tail warps read it while the large products run
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {  // columns 448.. : 7 K-blocks into the tile
      uint64_t pd, vd;
      pv_desc(j, ks, pd, vd);
      tc::mma_bf16(tmem + kColS + kTok * b, pd, vd + 7 * (kKvBlock >> 4), id_vt, ks > 0);
    }
    tc::commit(&ctl.tail_full[b]);
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint64_t pd, vd;
      pv_desc(j, ks, pd, vd);
      tc::mma_bf16(tmem + 0, pd, vd, id_v0, j > 0 || ks > 0);
      tc::mma_bf16(tmem + 256, pd, vd + 4 * (kKvBlock >> 4), id_v1, j > 0 || ks > 0);
    }
  };
  auto pv_second_round = [&](int j) {
    const int b = j & 1;
    tc::mbar_wait(&ctl.tail_empty, j & 1, abort, a.status);  // every tail warp has read round one
    tc::fence_after_sync();
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {  // columns 480.. : 64 bytes further into the swizzle atom
      uint64_t pd, vd;
      pv_desc(j, ks, pd, vd);
      tc::mma_bf16(tmem + kColS + kTok * b, pd, vd + (7 * (kKvBlock >> 4) + 4), id_vt, ks > 0);
    }
    tc::commit(&ctl.tail_full[b]);
    tc::commit(&ctl.kv_empty[b]);
    tc::commit(&ctl.p_free);
  };

  if (warp == kWarpQK || warp == kWarpQK + 1) {
    // ---------------- Q K^T issuers ----------------
    // warp kWarpQK + b issues the tiles j = b (mod 2), from lane 0: one thread issues an MMA
    // only every ~55 cycles and two lanes of one warp take turns, while two warps keep the
    // tensor core's operand reads busy.  Each warp owns one S buffer and one KV buffer, so
    // every barrier it waits on keeps a single waiter and its operands stay fixed.
    const int b = warp - kWarpQK;
    if (lane == 0) {
      if (b == 0) {
        tc::prefetch_tmap(&qmap);
        tc::mbar_arrive_expect_tx(&ctl.q_full, kQBytes);
        for (int kb = 0; kb < 9; ++kb) tc::tma_load_3d(s_q + kb * kQBlock, &qmap, kb * 64, 0, t, &ctl.q_full);
      }
      const uint32_t id_qk = tc::idesc_bf16(kTok, false, false);
      tc::mbar_wait(&ctl.q_full, 0, abort, a.status);
      // descriptors advance by adding (byte offset >> 4) to the start-address field
      const uint64_t qd0 = tc::desc_kmajor_sw128(smem_u32(s_q));
      const uint64_t kd = tc::desc_kmajor_sw128(smem_u32(s_kv + b * kKvBytes));
      const uint32_t d = tmem + kColS + kTok * b;
      for (int j = b; j < nt; j += 2) {
        // S = Q K^T of tile j into S buffer b
        tc::mbar_wait(&ctl.kv_full[b], (j >> 1) & 1, abort, a.status);
        tc::mbar_wait(&ctl.s_free[b], ((j >> 1) & 1) ^ 1, abort, a.status);
        tc::fence_after_sync();
#pragma unroll
        for (int st = 0; st < 36; ++st) {
          const uint32_t kb = st >> 2, k = st & 3;
          tc::mma_bf16(d, qd0 + (kb * (kQBlock >> 4) + 2 * k), kd + (kb * (kKvBlock >> 4) + 2 * k), id_qk, st > 0);
        }
        tc::commit(&ctl.s_full[b]);
        tc::commit(&ctl.kv_empty[b]);
      }
    }
    __syncwarp();
  } else if (warp >= kWarpSoft0 && warp < kWarpSoft0 + 4) {
    // ---------------- S -> P (warps 4..7) ----------------
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;  // head row
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = a.sm_scale * 1.4426950408889634f;  // logits in log2 units
    // l sums the bf16-rounded weights that the P V product uses (it normalises O);
    // lx sums the unrounded weights (it gives the log-sum-exp)
    float m_ref = -INFINITY, l = 0.f, lx = 0.f;
    // lane 0 of warp 4 issues every P V (see pv_main, pv_second_round)
    const bool pv = warp == kWarpSoft0 && lane == 0;
    for (int j = 0; j < nt; ++j) {
      const int b = j & 1;
      if (pv && j > 0) pv_second_round(j - 1);
      __syncwarp();
      // the gather warps flag the tile's real entries before they release the buffer
      tc::mbar_wait(&ctl.kv_full[b], (j >> 1) & 1, abort, a.status);
      const uint32_t mask = __ballot_sync(0xffffffffu, ctl.valid[b][lane] != 0);
      tc::mbar_wait(&ctl.s_full[b], (j >> 1) & 1, abort, a.status);
      tc::fence_after_sync();
      uint32_t sr[32];
      tc::tmem_ld32(tmem + lane_base + kColS + kTok * b, sr);
      tc::tmem_wait_ld();
      float x[32];
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        x[i] = ((mask >> i) & 1u) ? __uint_as_float(sr[i]) * c2 : -INFINITY;
        mt = fmaxf(mt, x[i]);
      }
      const bool need = mt > m_ref + kRescaleLog2 || (m_ref == -INFINITY && mt > -INFINITY);
      const float m_new = need ? mt : m_ref;
      const float alpha = need ? fast_exp2(m_ref - m_new) : 1.f;  // 2^-inf = 0
      // the tail warps rescale their part of the accumulator with the same max
      s_m[b * 128 + m] = m_new;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&ctl.m_ready[b]);
      // the weights need only the new max: they are formed while the previous tile's
      // products may still be running
      uint32_t pk[16];
      float lsum = 0.f, lxsum = 0.f;
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float p0 = (m_new == -INFINITY) ? 0.f : fast_exp2(x[i] - m_new);
        const float p1 = (m_new == -INFINITY) ? 0.f : fast_exp2(x[i + 1] - m_new);
        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
        lsum += __low2float(pb) + __high2float(pb);
        lxsum += p0 + p1;
        pk[i >> 1] = *reinterpret_cast<const uint32_t*>(&pb);
      }
      // every P V product of the previous tile has completed: P may be overwritten and the
      // TMEM accumulator rescaled
      if (j > 0) tc::mbar_wait(&ctl.p_free, (j - 1) & 1, abort, a.status);
      tc::fence_after_sync();
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        for (int c = 0; c < kVLeft; c += 16) {
          uint32_t r[16];
          tc::tmem_ld16(tmem + lane_base + c, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tc::tmem_st16(tmem + lane_base + c, r);
        }
        tc::tmem_wait_st();
      }
      l = l * alpha + lsum;
      lx = lx * alpha + lxsum;
      m_ref = m_new;
      // P row m: core matrix (m/8, chunk c) at (m/8)*512 + c*128, row offset (m%8)*16
      uint8_t* prow = s_p + (m >> 3) * 512 + (m & 7) * 16;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(prow + c * 128) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      tc::fence_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&ctl.p_full);
      if (pv) pv_main(j);
      __syncwarp();
    }
    if (pv && nt > 0) pv_second_round(nt - 1);
    __syncwarp();
    // every product has completed; hand (max, sums) to the tail warps through the P buffer
    if (nt > 0) tc::mbar_wait(&ctl.p_free, (nt - 1) & 1, abort, a.status);
    tc::fence_after_sync();
    float* s_fin = reinterpret_cast<float*>(s_p);  // [3][128]
    s_fin[m] = m_ref;
    s_fin[128 + m] = l;
    s_fin[256 + m] = lx;
    asm volatile("bar.sync 1, 256;" ::: "memory");  // S -> P and tail warps
    // (the TMEM columns are written by every warp after the role loops; see below)
  } else if (warp >= kWarpTail0 && warp < kWarpTail0 + 4) {
    // ---------------- tail rounds (warps 8..11): output columns 448..511 ----------------
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    float m_prev = -INFINITY;
    float ot[kVTail];
#pragma unroll
    for (int i = 0; i < kVTail; ++i) ot[i] = 0.f;
    for (int j = 0; j < nt; ++j) {
      const int b = j & 1;
      // the running max the S -> P warps used for this tile: rescale by the same factor
      tc::mbar_wait(&ctl.m_ready[b], (j >> 1) & 1, abort, a.status);
      const float m_new = s_m[b * 128 + m];
      const float alpha = (m_new == m_prev) ? 1.f : fast_exp2(m_prev - m_new);  // 2^-inf = 0
      m_prev = m_new;
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int i = 0; i < kVTail; ++i) ot[i] *= alpha;
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        tc::mbar_wait(&ctl.tail_full[b], r, abort, a.status);
        tc::fence_after_sync();
        uint32_t rr[32];
        tc::tmem_ld32(tmem + lane_base + kColS + kTok * b, rr);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) ot[32 * r + i] += __uint_as_float(rr[i]);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(r == 0 ? &ctl.tail_empty : &ctl.s_free[b]);
      }
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");  // (max, sums) from the S -> P warps
    const float* s_fin = reinterpret_cast<const float*>(s_p);
    const float m_ref = s_fin[m], l = s_fin[128 + m], lx = s_fin[256 + m];
    // columns 448..511 into the staged output rows (written out below by every warp)
    {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint8_t* row = smem + kOffQ + m * kStagePitch + 2 * kVLeft;
#pragma unroll
      for (int c = 0; c < kVTail; c += 8)
        *reinterpret_cast<uint4*>(row + 2 * c) =
            make_uint4(pack_bf16(ot[c] * inv, ot[c + 1] * inv), pack_bf16(ot[c + 2] * inv, ot[c + 3] * inv),
                       pack_bf16(ot[c + 4] * inv, ot[c + 5] * inv), pack_bf16(ot[c + 6] * inv, ot[c + 7] * inv));
    }
    (void)m_ref;
    (void)lx;
  } else {
    // ---------------- gather + dequantise (warps 2, 3, 12..15) ----------------
    // Thread g owns entry tok = g / 6 of every tile and its 16-byte code chunks
    // c = s, s + 6, .., s + 30 (s = g % 6): one index -> page -> record lookup per tile, and
    // six threads read one record's 576 codes in contiguous 96-byte runs.  The loads run
    // ahead of their use: while tile j is converted, the index entry of tile j + 4, the page
    // of tile j + 3, an L2 prefetch of the records of tile j + 2 and the codes of tile j + 1
    // are in flight, so no iteration waits on a load it issued itself and the code loads
    // find their lines in L2.
    static_assert(kTok * 6 == 32 * kGatherWarps && kChunks == 36, "six threads per entry, six chunks each");
    const int g = (warp < 4 ? warp - 2 : warp - 10) * 32 + lane;  // 0..191
    const int tok = g / 6, s6 = g % 6;
    const bool reporter = s6 == 0;              // one thread per entry reports bad input
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
    uint4 code[6];
    float scl[6];
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
      for (int k = 0; k < 6; ++k) {
        code[k] = make_uint4(0u, 0u, 0u, 0u);
        scl[k] = 0.f;
      }
      if (rec) {
        live = true;
#pragma unroll
        for (int k = 0; k < 6; ++k) {
          const int c = s6 + 6 * k;
          asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(code[k].x), "=r"(code[k].y), "=r"(code[k].z), "=r"(code[k].w)
                       : "l"(rec + 16 * c));
          asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];"
                       : "=f"(scl[k]) : "l"(rec + kKvScaleOff + 4 * (c >> 3)));
        }
      }
    };
    // pull the record of the entry at position p on page pg towards L2 (the six threads of
    // the entry take one 128-byte line each; together they cover the 608-byte record)
    auto prefetch_record = [&](int p, int pg) {
      if (in_range(p) && pg >= 0 && pg < a.num_pages) {
        const uint8_t* rec = a.kv_cache + (static_cast<int64_t>(pg) * kPage + p % kPage) * kKvTokBytes;
        asm volatile("prefetch.global.L2 [%0];" :: "l"(rec + min(128 * s6, kKvTokBytes - 1)));
      }
    };
    // warm L2 with this split's index entries and the sequence's page-table row (one
    // 128-byte line per thread), so that the first lookups do not each pay a DRAM access
    {
      const int e_lo = tile0 * kTok, e_hi = min(a.topk, (tile0 + nt) * kTok);
      const int npg = min(a.max_pages, (L + kPage - 1) / kPage);
      if (e_lo + 32 * g < e_hi) asm volatile("prefetch.global.L2 [%0];" :: "l"(idx + e_lo + 32 * g));
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
      const int b = j & 1;
      uint8_t* kv = s_kv + b * kKvBytes;
      // requests for the tiles ahead: the index of j + 4, the page of j + 3 and the record of
      // j + 2 (towards L2) now, the codes of j + 1 once this tile's have left their registers
      const int p4n = entry(j + 4);
      const int pg3n = page_of(p3);
      prefetch_record(p2, pg2);
      // this tile's codes -> bf16 in registers
      uint4 o0s[6], o1s[6];
      const bool live_j = live;
#pragma unroll
      for (int k = 0; k < 6; ++k) {
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
      tc::mbar_wait(&ctl.kv_empty[b], ((j >> 1) & 1) ^ 1, abort, a.status);
#pragma unroll
      for (int k = 0; k < 6; ++k) {
        const int c = s6 + 6 * k;
        const int kb = c >> 2, cc = (c & 3) * 2;
        uint8_t* row = kv + kb * kKvBlock + tok * 128;
        *reinterpret_cast<uint4*>(row + ((cc ^ (tok & 7)) << 4)) = o0s[k];
        *reinterpret_cast<uint4*>(row + (((cc + 1) ^ (tok & 7)) << 4)) = o1s[k];
      }
      if (reporter) ctl.valid[b][tok] = live_j ? 1 : 0;
      tc::fence_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&ctl.kv_full[b]);
    }
  }
  // ---- the output rows, normalised, as bf16: to the output (one split) or to the
  // workspace (several splits; merged by sfa_combine_kernel).  Columns 0..447 come from
  // TMEM: warp w reads its lane quadrant (w mod 4), columns 112 (w / 4) .. +112, and stages
  // them in the (idle) Q buffer next to the tail warps' columns; then every warp writes
  // whole rows, 512 contiguous bytes per instruction. ----
  tc::fence_before_sync();
  __syncthreads();  // the S -> P warps have seen the last product complete and published (m, l, lx)
  tc::fence_after_sync();
  {
    const float* s_fin = reinterpret_cast<const float*>(s_p);  // [3][128]: max, l, lx
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float l = s_fin[128 + m];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint8_t* row = smem + kOffQ + m * kStagePitch;
    const int cbeg = 112 * (warp >> 2);
    for (int c = cbeg; c < cbeg + 112; c += 32) {
      uint32_t r[32];
      const int nc = min(32, cbeg + 112 - c);  // 32, 32, 32, 16
      if (nt > 0) {
        tc::tmem_ld16(tmem + lane_base + c, reinterpret_cast<uint32_t(&)[16]>(r[0]));
        if (nc > 16) tc::tmem_ld16(tmem + lane_base + c + 16, reinterpret_cast<uint32_t(&)[16]>(r[16]));
        tc::tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = 0u;
      }
#pragma unroll
      for (int i = 0; i < 32; i += 8) {
        if (i < nc)
          *reinterpret_cast<uint4*>(row + 2 * (c + i)) =
              make_uint4(pack_bf16(__uint_as_float(r[i]) * inv, __uint_as_float(r[i + 1]) * inv),
                         pack_bf16(__uint_as_float(r[i + 2]) * inv, __uint_as_float(r[i + 3]) * inv),
                         pack_bf16(__uint_as_float(r[i + 4]) * inv, __uint_as_float(r[i + 5]) * inv),
                         pack_bf16(__uint_as_float(r[i + 6]) * inv, __uint_as_float(r[i + 7]) * inv));
      }
    }
    if (m < a.h_s && warp >= kWarpSoft0 && warp < kWarpSoft0 + 4) {
      const float m_ref = s_fin[m], lx = s_fin[256 + m];
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
    // row h: 64 pieces of 16 bytes; thread i takes piece i % 64 of rows i / 64, + 8, ..
    const int piece = tid & 63;
    for (int h = tid >> 6; h < a.h_s; h += kThreads / 64) {
      __nv_bfloat16* dst = pl.nsplit == 1
                               ? static_cast<__nv_bfloat16*>(a.out) + (static_cast<size_t>(t) * a.h_s + h) * kVDim
                               : pl.ws_o + ((static_cast<size_t>(t) * pl.nsplit + split) * a.h_s + h) * kVDim;
      *reinterpret_cast<uint4*>(dst + 8 * piece) =
          *reinterpret_cast<const uint4*>(smem + kOffQ + h * kStagePitch + 16 * piece);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// Merge the splits of each (row, head).  Split s holds O_s / l_s with running max m_s; with
// M = max_s m_s and c_s = 2^(m_s - M) l_s the output is sum_s c_s (O_s / l_s) / sum_s c_s.
__global__ void __launch_bounds__(128)
sfa_combine_kernel(SfaArgs a, SfaPlan pl) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x, h = blockIdx.y;
  const int ns = pl.nsplit;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, pl.ws_ml[4 * ((static_cast<size_t>(t) * ns + s) * a.h_s + h)]);
  float csum = 0.f, wsum_x = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < ns; ++s) {
    const size_t slot = (static_cast<size_t>(t) * ns + s) * a.h_s + h;
    const float4 ml = *reinterpret_cast<const float4*>(pl.ws_ml + 4 * slot);
    const float wgt = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
    const float c = wgt * ml.y;
    csum += c;
    wsum_x += wgt * ml.z;
    const uint2 v = *reinterpret_cast<const uint2*>(pl.ws_o + slot * kVDim + 4 * threadIdx.x);
    const __nv_bfloat162 v01 = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
    const __nv_bfloat162 v23 = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
    acc[0] += c * __low2float(v01); acc[1] += c * __high2float(v01);
    acc[2] += c * __low2float(v23); acc[3] += c * __high2float(v23);
  }
  const float inv = csum > 0.f ? 1.f / csum : 0.f;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (static_cast<size_t>(t) * a.h_s + h) * kVDim;
  *reinterpret_cast<uint2*>(out + 4 * threadIdx.x) =
      make_uint2(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv));
  if (a.out_lse && threadIdx.x == 0)
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
  const int ns = split_count(n_q, topk);
  if (ns <= 1) return 0;
  return ws_o_bytes(n_q, h_s, ns) + static_cast<size_t>(n_q) * ns * h_s * 4 * sizeof(float);
}

cudaError_t launch_sfa(const SfaArgs& a, cudaStream_t s, const char** err) {
  if (a.n_q == 0) return cudaSuccess;
  SfaPlan pl{};
  pl.nsplit = split_count(a.n_q, a.topk);
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
  e = launch_pdl(sfa_tc_kernel, dim3(pl.nsplit, a.n_q), dim3(kThreads), kSmemBytes, s, 1, qmap, a, pl);
  if (e != cudaSuccess || pl.nsplit == 1) return e;
  return launch_pdl(sfa_combine_kernel, dim3(a.n_q, a.h_s), dim3(128), 0, s, 1, a, pl);
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
