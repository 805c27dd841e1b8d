// Fused Lightning Indexer + Top-K on the 5th-generation tensor cores.
//
// "Deep Dive into Sparse Attention and Engineering Optimizations for Efficient Inference
// in Kimi K3.1 Pro", section 2.1, and "Kimi K3.1 Pro Inference Acceleration: Day0
// Optimization on Heterogeneous AI Hardware", section "Lightning Indexer Three-Stream
// Coordination": scoring, head-weight weighting and Top-K selection run in one kernel
// reading the paged K-cache directly, with Top-K pipelined behind the K-cache reads; the
// section "Full MXFP8 Quantization with Per-Group Dynamic Scaling for LI" gives the
// operand format (E4M3, one scale per 32 elements).
//
//   score[t, p] = sum_h w[t, h] * max(0, q_hat[t, h] . k_hat[p])
//
// One thread-block cluster of C CTAs handles a group of G query rows of one sequence;
// CTA r owns the r-th chunk (a multiple of 128 positions) of the positions the group may
// select.  Inside a CTA, warps specialise:
//   warp 0     producer: per 128-position tile, two TMA loads of 64x128 E4M3 page rows
//              (128-byte swizzle) and two 256-byte bulk loads of the pages' E8M0 scales
//              into an S-stage shared-memory ring, issued by two lanes in turn;
//   MMA warps  (two when N <= 128) each take every other tile: transpose the tile's
//              scales into the tcgen05 scale-factor layout, copy them to TMEM and issue four
//              block-scaled MXFP8 MMAs (M = 128 positions, N = G * Hp query heads,
//              K = 4 x 32) into their own TMEM accumulator;
//   epilogue   one set of four warps per accumulator: one TMEM lane (= one position) per
//              thread, ReLU, head weights and the sum over heads in registers; the score's
//              order-preserving key goes to shared memory and its top radix digit into a
//              histogram for the selection.  No score leaves the chip.
// The MXFP8 queries are quantised on chip into the MMA's B operand at kernel start.  After
// the scan, the cluster selects the Top-K of every row over distributed shared memory
// (topk_cluster.cuh).

#include <algorithm>
#include <mutex>
#include <cfloat>
#include <cuda.h>

#include "dsa_common.cuh"
#include "dsa_launch.h"
#include "quant_tok.cuh"
#include "tc_utils.cuh"
#include "topk_cluster.cuh"

namespace dsa {
namespace {

constexpr int kMaxAcc = 4;

// TMEM accumulators per CTA for N = G * HP query-head columns, MMA-issuing warps and
// epilogue sets.  Tile t goes to accumulator t mod acc_count, drained by epilogue set
// t mod acc_count (four warps, one per TMEM lane quarter) and issued by warp t mod
// mma_warps, so each set owns one accumulator and each issuer the accumulators of its
// residue.  A single thread can only issue a tcgen05.mma every ~120-200 cycles whatever N
// is, so two issuers are needed to keep up with the page stream.  The epilogue is a chain
// of TMEM loads, the head sum and the key and histogram stores per position: with N <= 64
// four sets (16 warps) hide its latencies where two cannot.  Each barrier that is waited on
// by parity must see its phases in order from one waiter, which is why an accumulator never
// moves between issuers and the ring has an even number of stages.
__host__ __device__ constexpr int mma_warps(int np) { return np <= 128 ? 2 : 1; }
__host__ __device__ constexpr int acc_count(int np) { return np <= 64 ? 4 : mma_warps(np); }
// warps: the producer, the MMA issuers, the epilogue sets, and one warp that writes a decode
// step's new tokens (fused writes) and otherwise only helps with the query quantisation
__host__ __device__ constexpr int threads_for(int np) { return 32 * (2 + mma_warps(np) + 4 * acc_count(np)); }
__host__ __device__ constexpr int writer_warp(int np) { return 1 + mma_warps(np) + 4 * acc_count(np); }
constexpr int kTileP = 128;            // positions per MMA tile = two pages
constexpr int kStageA = kTileP * kIdxDim;        // 16384 B of E4M3 codes
constexpr int kStageSF = kTileP * 4;             // 512 B of E8M0 scales (position order)
constexpr int kStageBytes = kStageA + 2 * kStageSF;  // + transposed copy: 17408 = 17 KB
constexpr int kProd = 2;              // producer lanes (the ring size is a multiple of it)
constexpr int kMaxCluster = 16;
constexpr int kMaxStages = 8;
constexpr int kLptMaxGroups = 256;    // launches with more row groups keep the grid order
// The selector's scratch and its candidate list live in the copy ring once the scan is done,
// which leaves room for a deeper ring: the scratch at the start, the candidates after it.
constexpr int kTopkBytes = (static_cast<int>(sizeof(TopkSmem)) + 15) / 16 * 16;
static_assert(kTopkBytes < kProd * kStageBytes, "the smallest ring holds the selector's scratch");

struct Plan {
  int G, H, Hp, Np, nacc, stages, chunk_cap;
  int ranked;  // the launch runs in several waves: clusters take the row groups longest first
  int read_once;  // no more row groups than sequences: each K page is read by one cluster
  uint32_t tmem_cols, d_col[kMaxAcc], sfa_col[kMaxAcc], sfb_col;
  // dynamic shared memory offsets (from a 1024-byte aligned base)
  uint32_t off_stage, off_b, off_sfb, off_w, off_keys, off_hist0, off_pages, off_bar, total;
};

// Query heads padded to the MMA's N granularity: 16, 32 or 64 rows per query row.
__host__ __device__ constexpr int padded_heads(int h) { return h <= 16 ? 16 : (h <= 32 ? 32 : 64); }

struct Barriers {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t pages_ready;
  uint64_t tfull[kMaxAcc];
  uint64_t tempty[kMaxAcc];
  uint64_t drain[kMaxAcc];  // after an abort: the issuer's own MMAs have completed
  uint64_t tok_written;     // this CTA's new tokens are in the K-cache (fused writes)
  uint32_t tmem_base;
  int abort;
  int seq;
  int n_max;
  int n_sel[4];
  int tok_mine;             // bit j: this CTA writes row j's new token
  int tok_tile;             // the first of its tiles that holds one of them (or a large value)
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ inline Plan make_plan(int G, int H, int chunk_cap, int stages) {
  Plan p{};
  p.G = G;
  p.H = H;
  p.Hp = padded_heads(H);
  p.Np = G * p.Hp;
  p.nacc = acc_count(p.Np);
  p.stages = stages;
  p.chunk_cap = chunk_cap;
  uint32_t used = p.nacc * p.Np + 4 * p.nacc + 8 * mma_warps(p.Np);
  uint32_t cols = 32;
  while (cols < used) cols *= 2;
  p.tmem_cols = cols;
  for (int i = 0; i < kMaxAcc; ++i) {
    p.d_col[i] = i * p.Np;
    p.sfa_col[i] = p.nacc * p.Np + 4 * i;
  }
  p.sfb_col = p.nacc * p.Np + 4 * p.nacc;  // issuer i keeps its own copy at sfb_col + 8 i
  uint32_t o = 0;
  p.off_stage = o; o += stages * kStageBytes;
  p.off_b = o = align_up(o, 1024); o += p.Np * kIdxDim;
  p.off_sfb = o = align_up(o, 16); o += 2 * 512;
  p.off_w = o = align_up(o, 16); o += 4 * G * p.Hp;  // read as float4
  p.off_keys = o = align_up(o, 16); o += 4u * G * chunk_cap;
  p.off_hist0 = o; o += 4u * G * kHistBins;
  p.off_pages = o; o += 4u * (chunk_cap / kPage + 2);
  p.off_bar = o = align_up(o, 16); o += sizeof(Barriers);
  p.total = o;
  return p;
}

// Number of positions row group [row0, row0 + G) scans: the largest selectable count of its
// rows (0 for an invalid sequence; the kernel prologue reports bad inputs).
__device__ inline uint32_t group_scan_len(const IndexerArgs& a, int row0, int G) {
  const int seq = __ldcg(a.q_seq + row0);
  if (seq < 0 || seq >= a.n_seq) return 0u;
  int L = __ldcg(a.seq_lens + seq);
  L = L < 0 ? 0 : (L > a.max_ctx ? a.max_ctx : L);
  uint32_t n = 0;
  for (int j = 0; j < G; ++j) {
    long long v = static_cast<long long>(__ldcg(a.q_pos + row0 + j)) + 1;
    v = v < 0 ? 0 : (v > L ? L : v);
    n = max(n, static_cast<uint32_t>(v));
  }
  return n;
}

// MXFP8-quantise one 128-wide bf16 row (this lane's four values, already loaded) straight
// into the B operand (128-byte swizzled K-major row n) and return this lane's group
// exponent code (lanes 0, 8, 16, 24 hold groups 0..3).  Same OCP MX rule as the cache writer.
__device__ __forceinline__ uint32_t quant_row_to_b(uint2 raw, uint8_t* b_row_base, int n) {
  const int lane = threadIdx.x & 31;
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
  float x[4] = {__low2float(a), __high2float(a), __low2float(b), __high2float(b)};
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = mx_shared_exp(amax);
  const float inv = exp2i(-e);
  uint32_t codes = 0;
  if (amax > 0.f)
    codes = static_cast<uint32_t>(f32x2_to_e4m3x2(x[0] * inv, x[1] * inv)) |
            (static_cast<uint32_t>(f32x2_to_e4m3x2(x[2] * inv, x[3] * inv)) << 16);
  const int chunk = lane >> 2;  // 16-byte chunk of the 128-byte row
  *reinterpret_cast<uint32_t*>(b_row_base + n * 128 + ((chunk ^ (n & 7)) << 4) + (lane & 3) * 4) = codes;
  return static_cast<uint32_t>(e + 127);
}

template <int G, int HP>
__global__ void __launch_bounds__(threads_for(G * HP), 1)
indexer_tc_kernel(const __grid_constant__ CUtensorMap kmap, IndexerArgs a, Plan pl) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  Barriers& bs = *reinterpret_cast<Barriers*>(smem + pl.off_bar);
  TopkSmem& tk = *reinterpret_cast<TopkSmem*>(smem + pl.off_stage);  // used after the scan only
  uint8_t* s_b = smem + pl.off_b;
  uint32_t* s_sfb = reinterpret_cast<uint32_t*>(smem + pl.off_sfb);
  float* s_w = reinterpret_cast<float*>(smem + pl.off_w);
  uint32_t* s_keys = reinterpret_cast<uint32_t*>(smem + pl.off_keys);
  uint32_t* s_hist0 = reinterpret_cast<uint32_t*>(smem + pl.off_hist0);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int C = static_cast<int>(cluster_nctarank());
  const int H = pl.H, S = pl.stages;
  constexpr int Hp = HP, Np = G * HP;
  constexpr int kThreads = threads_for(Np), kMma = mma_warps(Np), kNacc = acc_count(Np);

  // ---- prologue -------------------------------------------------------------------
  for (int i = tid; i < G * kHistBins; i += kThreads) s_hist0[i] = 0;
  pdl_launch_dependents();
  // nothing global is read before the previous kernel on the stream is done, unless that
  // kernel is the cache writer of a decode step (early_inputs): then only the K-cache, the
  // writer's output, waits (the producer lanes, below); the reads before it bypass L1
  if (!a.early_inputs) pdl_wait();
  // Which row group this cluster takes: the groups in order of decreasing scan length (ties
  // in group order), so that when the grid runs in several waves the clusters of the
  // longest groups are dispatched first and the short ones fill in behind them.  Every CTA
  // of the cluster computes the same ranking.
  int group = static_cast<int>(blockIdx.y);
  const int n_groups = static_cast<int>(gridDim.y);
  if (pl.ranked && n_groups <= kLptMaxGroups) {
    uint32_t* s_len = reinterpret_cast<uint32_t*>(smem + pl.off_stage);  // the copy ring is idle yet
    for (int g = tid; g < n_groups; g += kThreads) s_len[g] = group_scan_len(a, g * G, G);
    __syncthreads();
    for (int g = tid; g < n_groups; g += kThreads) {
      const uint32_t v = s_len[g];
      int r = 0;
      for (int h = 0; h < n_groups; ++h) {
        const uint32_t u = s_len[h];
        r += (u > v || (u == v && h < g)) ? 1 : 0;
      }
      if (r == static_cast<int>(blockIdx.y)) s_len[kLptMaxGroups] = static_cast<uint32_t>(g);
    }
    __syncthreads();
    group = static_cast<int>(s_len[kLptMaxGroups]);
  }
  const int row0 = group * G;
  if (warp == 2) {
    // while thread 0 reads the sequence information below (a chain of dependent loads),
    // this warp pulls the next links of that chain and the sequence's page-table row towards
    // L2 (one 128-byte line per lane), so that only the first load of each chain pays a DRAM
    // access: the sequence lengths and the rows' positions, then the page-table row
    for (int i = 32 * lane; i < a.n_seq && i < 32 * 32 * 4; i += 32 * 32)
      asm volatile("prefetch.global.L2 [%0];" :: "l"(a.seq_lens + i));
    if (lane == 0) asm volatile("prefetch.global.L2 [%0];" :: "l"(a.q_pos + row0));
    if (lane == 1 && G > 1) asm volatile("prefetch.global.L2 [%0];" :: "l"(a.q_pos + row0 + G - 1));
    const int sq = __ldcg(a.q_seq + row0);
    if (sq >= 0 && sq < a.n_seq) {
      const int32_t* prow = a.page_table + static_cast<size_t>(sq) * a.max_pages;
      for (int i = 32 * lane; i < a.max_pages && i < 32 * 32 * 4; i += 32 * 32)
        asm volatile("prefetch.global.L2 [%0];" :: "l"(prow + i));
    }
  }
  if (tid == 0) {
    int seq = __ldcg(a.q_seq + row0);
    unsigned bad = 0;
    if (seq < 0 || seq >= a.n_seq) { bad |= DSA_STATUS_BAD_SEQ; seq = -1; }
    int L = 0;
    if (seq >= 0) {
      L = __ldcg(a.seq_lens + seq);
      if (L < 0 || L > a.max_ctx) { bad |= DSA_STATUS_BAD_LEN; L = L < 0 ? 0 : a.max_ctx; }
    }
    int n_max = 0;
    for (int j = 0; j < G; ++j) {
      if (__ldcg(a.q_seq + row0 + j) != seq && seq >= 0) bad |= DSA_STATUS_BAD_SEQ;
      long long n = static_cast<long long>(__ldcg(a.q_pos + row0 + j)) + 1;
      n = n < 0 ? 0 : (n > L ? L : n);
      bs.n_sel[j] = static_cast<int>(n);
      n_max = n > n_max ? static_cast<int>(n) : n_max;
    }
    bs.seq = seq;
    bs.n_max = n_max;
    bs.abort = 0;
    // fused writes: row j's new token (at its own position) is written by the CTA whose
    // chunk holds that position, before the tile that holds it is loaded; a token outside
    // every chunk (its row selects nothing there) goes to the last CTA
    int mine = 0, tok_tile = 1 << 30;
    if (a.fuse_writes) {
      int chk = (n_max + C - 1) / C;
      chk = (chk + kTileP - 1) / kTileP * kTileP;
      if (chk > pl.chunk_cap) chk = pl.chunk_cap;
      for (int j = 0; j < G; ++j) {
        const int p = __ldcg(a.q_pos + row0 + j);
        const bool scanned = p >= 0 && p < n_max && chk > 0;
        const int owner = scanned ? min(p / chk, C - 1) : C - 1;
        if (owner == rank) {
          mine |= 1 << j;
          if (scanned) tok_tile = min(tok_tile, (p - rank * chk) / kTileP);
        }
      }
    }
    bs.tok_mine = mine;
    bs.tok_tile = tok_tile;
    tc::mbar_init(&bs.tok_written, static_cast<uint32_t>(max(1, __popc(mine))));
    if (bad && rank == 0) flag(a.status, bad);
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&bs.full[s], 1);
      tc::mbar_init(&bs.empty[s], 1);
    }
    tc::mbar_init(&bs.pages_ready, 32);
    for (int i = 0; i < kNacc; ++i) {
      tc::mbar_init(&bs.tfull[i], 1);
      tc::mbar_init(&bs.tempty[i], 128);
      tc::mbar_init(&bs.drain[i], 1);
    }
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(&bs.tmem_base, pl.tmem_cols);
  tc::fence_before_sync();
  __syncthreads();  // barriers, sequence info and the TMEM base are visible to every warp
  tc::fence_after_sync();

  const int seq = bs.seq;
  const int n_max = bs.n_max;
  int chunk = (n_max + C - 1) / C;
  chunk = (chunk + kTileP - 1) / kTileP * kTileP;
  if (chunk > pl.chunk_cap) chunk = pl.chunk_cap;
  const int c0 = rank * chunk;
  const int len = max(0, min(chunk, n_max - c0));
  const int ntiles = (len + kTileP - 1) / kTileP;
  const int n_pages_needed = (n_max + kPage - 1) / kPage;
  const int32_t* ptab = a.page_table + static_cast<size_t>(seq < 0 ? 0 : seq) * a.max_pages;
  const uint32_t tmem = bs.tmem_base;
  volatile int* abort = &bs.abort;
  const uint64_t wait_ns = a.wait_ns;

  auto phys_page = [&](int lp) -> int {
    if (seq < 0 || lp >= n_pages_needed || lp >= a.max_pages) return -1;
    const int pg = __ldcg(ptab + lp);
    return (pg >= 0 && pg < a.num_pages) ? pg : -2;
  };
  // physical page of each of this chunk's logical pages (-1 past the end, -2 invalid),
  // looked up once by the producer warp: s_pages[i] belongs to logical page c0/64 + i
  int32_t* s_pages = reinterpret_cast<int32_t*>(smem + pl.off_pages);

  if (warp == 0) {
    // ---------------- producer: starts streaming pages while the others prepare ----------------
    for (int i = lane; i < 2 * ntiles; i += 32) s_pages[i] = phys_page(c0 / kPage + i);
    __syncwarp();
    tc::mbar_arrive(&bs.pages_ready);
    if (lane < kProd) {
      if (a.early_inputs) pdl_wait();  // the K-cache copies follow the cache writer
      // lane l issues tiles t = l (mod kProd): one thread alone cannot issue copies fast
      // enough to keep the HBM busy, and with a ring of a multiple of kProd stages each
      // stage keeps one issuer
      if (lane == 0) tc::prefetch_tmap(&kmap);
      // pages that no other cluster reads are streamed evict-first: a stream larger than L2
      // would otherwise evict the kernel's own instructions and the other inputs
      const uint64_t pol = pl.read_once ? tc::l2_policy_evict_first() : tc::l2_policy_evict_normal();
      int last = -1;  // the last tile this lane issued
      for (int t = a.stall_producer ? ntiles : lane; t < ntiles; t += kProd) {
        const int s = t % S, it = t / S;
        if (!tc::mbar_wait(&bs.empty[s], (it & 1) ^ 1, abort, a.status, wait_ns)) break;
        // a tile holding this CTA's new token is loaded only after the token is written
        if (t >= bs.tok_tile && !tc::mbar_wait(&bs.tok_written, 0, abort, a.status, wait_ns)) break;
        uint8_t* st = smem + pl.off_stage + s * kStageBytes;
        const int pg0 = s_pages[2 * t], pg1 = s_pages[2 * t + 1];
        if (pg0 == -2 || pg1 == -2) flag(a.status, DSA_STATUS_BAD_PAGE);
        const uint32_t bytes = (pg0 >= 0 ? (kKPageBytes) : 0) + (pg1 >= 0 ? (kKPageBytes) : 0);
        tc::mbar_arrive_expect_tx(&bs.full[s], bytes);
        if (pg0 >= 0) {
          tc::tma_load_3d_hint(st, &kmap, 0, 0, pg0, &bs.full[s], pol);
          tc::bulk_load_hint(st + kStageA, a.k_cache + static_cast<int64_t>(pg0) * kKPageBytes + kKScaleOff, 256,
                             &bs.full[s], pol);
        }
        if (pg1 >= 0) {
          tc::tma_load_3d_hint(st + kStageA / 2, &kmap, 0, 0, pg1, &bs.full[s], pol);
          tc::bulk_load_hint(st + kStageA + 256, a.k_cache + static_cast<int64_t>(pg1) * kKPageBytes + kKScaleOff, 256,
                             &bs.full[s], pol);
        }
        last = t;
      }
      if (*abort) {
        // copies may still be landing in the ring: wait for the newest phase of each stage
        // this lane filled.  Its last S / kProd tiles sit in distinct stages (a lane's tiles
        // are kProd apart and S is a multiple of kProd) that no other lane uses.
        for (int t = last; t >= 0 && t > last - S; t -= kProd) tc::mbar_drain(&bs.full[t % S], (t / S) & 1, wait_ns);
      }
    }
  } else {
    // ---------------- warps 1..9: B operand, head weights, then MMA / epilogue ----------------
    // On-chip MXFP8 quantisation of the group's queries (row n = j * Hp + h), with each
    // warp's row loads issued together before they are used.
    constexpr int kPrepWarps = kThreads / 32 - 1;
    constexpr int kBatch = 8;
    const __nv_bfloat16* qbase = static_cast<const __nv_bfloat16*>(a.q);
    // the head weights are requested first, so that their loads share the round trip of the
    // query rows' loads below
    constexpr int kWPer = (Np + kThreads - 33) / (kThreads - 32);
    float wv[kWPer];
#pragma unroll
    for (int r = 0; r < kWPer; ++r) {
      const int i = tid - 32 + r * (kThreads - 32), j = i / Hp, h = i % Hp;
      wv[r] = (i < G * Hp && h < H) ? __ldcg(a.w + static_cast<size_t>(row0 + j) * H + h) : 0.f;
    }
    for (int n0 = warp - 1; n0 < Np; n0 += kPrepWarps * kBatch) {
      uint2 raw[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int n = n0 + k * kPrepWarps;
        raw[k] = make_uint2(0u, 0u);
        if (n < Np && (n % Hp) < H)
          raw[k] = __ldcg(reinterpret_cast<const uint2*>(qbase + (static_cast<size_t>(row0 + n / Hp) * H + (n % Hp)) * kIdxDim +
                                                         4 * lane));
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int n = n0 + k * kPrepWarps;
        if (n >= Np) break;
        const uint32_t ecode = quant_row_to_b(raw[k], s_b, n);  // padding rows: zero codes, code 127
        // gather the four group codes (lanes 0, 8, 16, 24) into one scale word
        const uint32_t e1 = __shfl_sync(0xffffffffu, ecode, 8), e2 = __shfl_sync(0xffffffffu, ecode, 16),
                       e3 = __shfl_sync(0xffffffffu, ecode, 24);
        if (lane == 0) {
          // scale-factor layout: block n/128, row n%32, word (n/32)%4
          s_sfb[(n >> 7) * 128 + (n & 31) * 4 + ((n >> 5) & 3)] = ecode | (e1 << 8) | (e2 << 16) | (e3 << 24);
        }
      }
    }
    // scale words of padding rows up to the end of the last 128-row block
    for (int n = Np + tid - 32; n < ((Np + 127) / 128) * 128; n += kThreads - 32)
      s_sfb[(n >> 7) * 128 + (n & 31) * 4 + ((n >> 5) & 3)] = 0x7F7F7F7Fu;
#pragma unroll
    for (int r = 0; r < kWPer; ++r) {
      const int i = tid - 32 + r * (kThreads - 32);
      if (i < G * Hp) s_w[i] = wv[r];
    }
    tc::fence_async_smem();
    asm volatile("bar.sync 1, %0;" :: "r"(kThreads - 32) : "memory");  // every warp but the producer
  }
  if (warp >= 1 && warp <= kMma) {
    // ---------------- MMA issuers: warp 1 + i takes tiles t = i (mod kMma) ----------------
    const int mi = warp - 1;
    const uint32_t sfb = tmem + pl.sfb_col + 8 * mi;
    if (lane == 0) {
      // each issuer copies the query scale factors to its own columns: its MMAs follow its
      // own copies in issue order
      tc::cp_32x128b_warpx4(sfb, tc::desc_sf_block(smem_u32(s_sfb)));
      if (Np > 128) tc::cp_32x128b_warpx4(sfb + 4, tc::desc_sf_block(smem_u32(s_sfb + 128)));
    }
    const uint64_t bdesc = tc::desc_kmajor_sw128(smem_u32(s_b));
    for (int t = mi; t < ntiles; t += kMma) {
      const int s = t % S, it = t / S;
      const int acc = t % kNacc, ia = t / kNacc;
      uint8_t* st = smem + pl.off_stage + s * kStageBytes;
      // (every lane waits; the warp leaves the loop together once a wait gives up)
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&bs.full[s], it & 1, abort, a.status, wait_ns))) break;
      // scales: position order -> [32 rows][4 words], word (i, j) = position 32 j + i
      const uint32_t* sf_nat = reinterpret_cast<const uint32_t*>(st + kStageA);
      uint32_t* sf_t = reinterpret_cast<uint32_t*>(st + kStageA + kStageSF);
      const uint4 v = make_uint4(sf_nat[lane], sf_nat[32 + lane], sf_nat[64 + lane], sf_nat[96 + lane]);
      *reinterpret_cast<uint4*>(sf_t + 4 * lane) = v;
      tc::fence_async_smem();
      __syncwarp();
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&bs.tempty[acc], (ia & 1) ^ 1, abort, a.status, wait_ns))) break;
      tc::fence_after_sync();
      if (lane == 0) {
        const uint32_t d = tmem + pl.d_col[acc];
        const uint32_t sfa = tmem + pl.sfa_col[acc];
        tc::cp_32x128b_warpx4(sfa, tc::desc_sf_block(smem_u32(sf_t)));
        const uint64_t adesc = tc::desc_kmajor_sw128(smem_u32(st));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_mxf8(d, adesc + 2 * k, bdesc + 2 * k, tc::idesc_mxf8_e4m3(Np, k), sfa, sfb, k > 0);
        tc::commit(&bs.empty[s]);
        tc::commit(&bs.tfull[acc]);
      }
      __syncwarp();
    }
    if (*abort && lane == 0) {
      // the epilogue no longer waits for this issuer's products: wait for them here
      tc::commit(&bs.drain[mi]);
      tc::mbar_drain(&bs.drain[mi], 0, wait_ns);
    }
    __syncwarp();
  } else if (warp == writer_warp(Np)) {
    // ---------------- fused writes: this CTA's share of the step's new tokens ----------------
    // row e's token, if this CTA owns it, with the same quantisers as the writer kernels;
    // the stores are made visible to the copy engine before the producer is signalled
    for (int e = 0; e < G; ++e) {
      if ((bs.tok_mine >> e) & 1) {
        const int64_t i = row0 + e;
        if (lane == 0 && seq >= 0) {
          // the contract: token i sits at row i's own position (its scan sees it)
          const int p = __ldcg(a.q_pos + i);
          const int64_t own = (p >= 0 && p / kPage < a.max_pages)
                                  ? static_cast<int64_t>(__ldcg(ptab + p / kPage)) * kPage + p % kPage
                                  : -1;
          if (own != __ldcg(a.slot_mapping + i)) flag(a.status, DSA_STATUS_BAD_PAGE);
        }
        const KTok kt = load_k_token(static_cast<const __nv_bfloat16*>(a.k_new), a.slot_mapping, i);
        const KvTok vt = load_kv_token(static_cast<const __nv_bfloat16*>(a.kv_new), a.slot_mapping, i);
        store_k_token(kt, const_cast<uint8_t*>(a.k_cache), a.num_slots, a.status);
        store_kv_token(vt, a.kv_cache, a.num_slots, a.status);
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bs.tok_written);
      }
    }
  } else if (warp > kMma) {
    // ---------------- epilogue: set i (four warps) drains accumulator i ----------------
    const int set = (warp - 1 - kMma) >> 2;    // which accumulator this warp drains
    const int quarter = warp & 3;              // TMEM lanes 32*quarter .. +31
    const int m = quarter * 32 + lane;         // tile row = position offset in the tile
    tc::mbar_wait(&bs.pages_ready, 0, abort, a.status, wait_ns);
    for (int t = set; t < ntiles; t += kNacc) {
      const int acc = t % kNacc, ia = t / kNacc;
      const bool ok = tc::mbar_wait(&bs.tfull[acc], ia & 1, abort, a.status, wait_ns);
      tc::fence_after_sync();
      const int local = t * kTileP + m;
      const int p = c0 + local;
      const bool page_ok = s_pages[local / kPage] >= 0;
      float sc[G];
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const uint32_t col = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + pl.d_col[acc] + j * HP;
        // the weights are read four at a time (one 16-byte shared load for four heads):
        // with a load per head the shared-memory pipe, not the arithmetic, set the pace
        const float4* w4 = reinterpret_cast<const float4*>(s_w + j * HP);
        float s4[4] = {0.f, 0.f, 0.f, 0.f};  // four independent chains over the heads
        // with four epilogue sets the heads come in halves of 32 TMEM columns (the larger
        // block has fewer registers per thread)
        constexpr int kPart = (kNacc > 2 && HP > 32) ? 32 : HP;
#pragma unroll
        for (int h1 = 0; h1 < HP; h1 += kPart) {
          uint32_t r[kPart];
#pragma unroll
          for (int h0 = 0; h0 < kPart; h0 += 16)
            tc::tmem_ld16(col + h1 + h0, reinterpret_cast<uint32_t(&)[16]>(r[h0]));
          tc::tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < kPart; h += 4) {
            const float4 w = w4[(h1 + h) >> 2];
            s4[0] = fmaf(w.x, relu_nan(__uint_as_float(r[h])), s4[0]);
            s4[1] = fmaf(w.y, relu_nan(__uint_as_float(r[h + 1])), s4[1]);
            s4[2] = fmaf(w.z, relu_nan(__uint_as_float(r[h + 2])), s4[2]);
            s4[3] = fmaf(w.w, relu_nan(__uint_as_float(r[h + 3])), s4[3]);
          }
        }
        sc[j] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
      }
      tc::fence_before_sync();
      tc::mbar_arrive(&bs.tempty[acc]);
      bool nan_seen = false;
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const bool valid = ok && page_ok && local < len && p < bs.n_sel[j];
        const uint32_t key = valid ? score_key(sc[j]) : 0u;
        nan_seen |= key == kNanKey;
        s_keys[j * pl.chunk_cap + local] = key;
        hist_add_top_digit(s_hist0 + j * kHistBins, key);
        if (a.out_full && valid) a.out_full[static_cast<size_t>(row0 + j) * a.max_ctx + p] = sc[j];
      }
      if (__any_sync(0xffffffffu, nan_seen) && lane == 0) flag(a.status, DSA_STATUS_NAN_SCORE);
    }
  }
  tc::fence_before_sync();
  __syncthreads();  // the ring is idle: every copy into it has landed, every MMA has read it
  topk_init(tk);
  cluster_sync();  // every CTA of the cluster has initialised its selector before DSMEM traffic

  if (a.out_idx) {
    // the copy ring is idle now: after the selector's scratch it holds the candidate lists
    uint2* cand = reinterpret_cast<uint2*>(smem + pl.off_stage + kTopkBytes);
    const int cand_cap = (pl.stages * kStageBytes - kTopkBytes) / static_cast<int>(sizeof(uint2));
#pragma unroll 1
    for (int j = 0; j < G; ++j) {
      const size_t row = static_cast<size_t>(row0 + j);
      cluster_topk_row(tk, s_keys + j * pl.chunk_cap, s_hist0 + j * kHistBins, c0, chunk, len, bs.n_sel[j], a.topk,
                       a.out_idx + row * a.topk, a.out_scores ? a.out_scores + row * a.topk : nullptr, cand, cand_cap,
                       j, a.status, wait_ns);
    }
  }
  // every CTA has waited for the writer before it leaves, so this grid never completes
  // before the writer does (the next kernel relies on that for the latent cache)
  if (a.early_inputs && tid == 0) pdl_wait();
  cluster_sync();  // no CTA leaves while its shared memory may still be addressed
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, pl.tmem_cols);
}

__global__ void fill_kernel(float* p, size_t n, float v) {
  pdl_launch_dependents();
  pdl_wait();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    p[i] = v;
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

// Clusters of c CTAs that fit on the GPU at once with one CTA per SM (the indexer's shared
// memory): the GPCs' SM counts are not multiples of most cluster sizes, so this is below
// n_sm / c (on a 152-SM part: 36 clusters of 4, 15 of 8, 8 of 12, 7 of 16).  Queried once
// per device and size, under a lock.
__global__ void cluster_fit_probe_kernel(int) {}
int clusters_that_fit(int c, int n_sm) {
  if (c <= 1) return n_sm;
  static std::mutex mu;
  static int cache[64][kMaxCluster + 1] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || c > kMaxCluster) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev][c]) return cache[dev][c];
  const int smem = 120 * 1024;
  if (cudaFuncSetAttribute(cluster_fit_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(cluster_fit_probe_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(c);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(c), 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, cluster_fit_probe_kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  cache[dev][c] = n;
  return n;
}

// Positions per CTA for a cluster of c CTAs over max_ctx positions.
inline int cap_for(int max_ctx, int c) {
  const int chunk = (max_ctx + c - 1) / c;
  return (chunk + kTileP - 1) / kTileP * kTileP;
}

// The cost of one row's selection, in positions scanned (about 10 us, the cluster Top-K).
constexpr int kSelectAllowance = 2048;

// Grid shape: rows per group and CTAs per cluster.
struct GridChoice {
  int G = 0, C = 0;
};

// The cluster size (1..16, any size) that gives the most CTAs while every group's cluster
// is resident at once, for groups of g rows; 0 if no size does (more groups than one wave).
int single_wave_cluster(int g, int n_q, int h_i, int max_ctx, int n_sm, size_t limit, long long* ctas) {
  const int n_groups = n_q / g;
  int best = 0;
  *ctas = 0;
  for (int c = 1; c <= kMaxCluster; ++c) {
    if (make_plan(g, h_i, cap_for(max_ctx, c), 4).total > limit) continue;
    if (clusters_that_fit(c, n_sm) < n_groups) continue;
    const long long n = static_cast<long long>(n_groups) * c;
    if (n > *ctas) {
      *ctas = n;
      best = c;
    }
  }
  return best;
}

GridChoice choose_grid(int q_group, int n_q, int h_i, int max_ctx, int n_sm, size_t limit) {
  GridChoice r;
  long long ctas = 0;
  const int C = single_wave_cluster(q_group, n_q, h_i, max_ctx, n_sm, limit, &ctas);
  // Few long row groups would leave most of the GPU idle even with the largest clusters:
  // scan the rows of a group one by one (each row its own cluster) when that puts more
  // CTAs to work; the shared reads of the group are then repeated, the selection is not.
  if (q_group > 1 && 2 * ctas < n_sm) {
    long long ctas1 = 0;
    const int C1 = single_wave_cluster(1, n_q, h_i, max_ctx, n_sm, limit, &ctas1);
    if (C1 && ctas1 > ctas) {
      r.G = 1;
      r.C = C1;
      return r;
    }
  }
  r.G = q_group;
  if (C) {
    r.C = C;
    return r;
  }
  // More groups than one wave holds: the grouping (the caller's, or one row per group) and
  // cluster size of least estimated time, waves x rows per group x (positions per CTA + an
  // allowance for each row's selection).  The scan's cost follows rows x positions (the
  // MMA's N and the epilogue grow with the rows of a group), so resident CTAs count more
  // than shared reads: prefill rows over a 64K prefix run 2.2x faster as single rows in
  // clusters of 4 (36 resident) than as groups of 4 in clusters of 16 (7 resident).
  double best = 0.0;
  for (int k = 0; k < (q_group > 1 ? 2 : 1); ++k) {
    const int g = k == 0 ? q_group : 1;
    const long long n_groups = n_q / g;
    for (int c = 1; c <= kMaxCluster; ++c) {
      if (make_plan(g, h_i, cap_for(max_ctx, c), 4).total > limit) continue;
      const int fit = clusters_that_fit(c, n_sm);
      if (fit < 1) continue;
      const long long waves = (n_groups + fit - 1) / fit;
      const double cost = static_cast<double>(waves) * g * (cap_for(max_ctx, c) + kSelectAllowance);
      if (!r.C || cost < best) {
        best = cost;
        r.G = g;
        r.C = c;
      }
    }
  }
  if (!r.C) {  // nothing fits (the launch reports it): the caller's grouping
    r.G = q_group;
    r.C = kMaxCluster;
  }
  return r;
}

template <int G, int HP>
cudaError_t launch_gh(const IndexerArgs& a, cudaStream_t s, const char** err, int C) {
  DevInfo di;
  if (!device_info(&di, err)) return cudaErrorInvalidDevice;
  const int n_groups = a.n_q / G;
  const size_t limit = static_cast<size_t>(di.smem_optin) - 1024;  // room for the 1024-byte alignment
  auto cap_for = [&](int c) { return dsa::cap_for(a.max_ctx, c); };
  int stages = kMaxStages;
  // a multiple of kProd (and so of the two MMA issuers): every stage keeps one issuer and
  // one waiter per barrier
  while (stages > kProd && make_plan(G, a.h_i, cap_for(C), stages).total > limit) stages -= kProd;
  Plan pl = make_plan(G, a.h_i, cap_for(C), stages);
  pl.ranked = n_groups > clusters_that_fit(C, di.n_sm) ? 1 : 0;
  pl.read_once = n_groups <= a.n_seq ? 1 : 0;
  if (pl.total > limit) {
    *err = "indexer: max_ctx too large for the on-chip score buffer";
    return cudaErrorInvalidValue;
  }
  // at least ~120 KB so that one CTA (and one TMEM allocation) owns each SM
  const size_t smem = std::max<size_t>(pl.total + 1024, 120 * 1024);

  EncodeFn enc = encode_fn();
  if (!enc) {
    *err = "indexer: cuTensorMapEncodeTiled is not available";
    return cudaErrorNotSupported;
  }
  CUtensorMap map;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kIdxDim), static_cast<cuuint64_t>(kPage),
                              static_cast<cuuint64_t>(a.num_pages)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kIdxDim), static_cast<cuuint64_t>(kKPageBytes)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kIdxDim), static_cast<cuuint32_t>(kPage), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(a.k_cache), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
    *err = "indexer: tensor map encoding failed";
    return cudaErrorInvalidValue;
  }
  auto kern = indexer_tc_kernel<G, HP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  if (a.out_full) {
    const size_t n = static_cast<size_t>(a.n_q) * a.max_ctx;
    e = launch_pdl(fill_kernel, dim3(1024), dim3(256), 0, s, 1, a.out_full, n, -INFINITY);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(kern, dim3(C, n_groups, 1), dim3(threads_for(G * HP)), smem, s, C, map, a, pl);
}

template <int G>
cudaError_t launch_g(const IndexerArgs& a, cudaStream_t s, const char** err, int C) {
  switch (padded_heads(a.h_i)) {
    case 16: return launch_gh<G, 16>(a, s, err, C);
    case 32: return launch_gh<G, 32>(a, s, err, C);
    default: return launch_gh<G, 64>(a, s, err, C);
  }
}

}  // namespace

cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t s, const char** err) {
  if (a.n_q == 0) return cudaSuccess;
  if (a.q_group < 1 || a.q_group > 4) {
    *err = "indexer: q_group must be 1..4";
    return cudaErrorInvalidValue;
  }
  DevInfo di;
  if (!device_info(&di, err)) return cudaErrorInvalidDevice;
  const GridChoice g = choose_grid(a.q_group, a.n_q, a.h_i, a.max_ctx, di.n_sm,
                                   static_cast<size_t>(di.smem_optin) - 1024);
  switch (g.G) {
    case 1: return launch_g<1>(a, s, err, g.C);
    case 2: return launch_g<2>(a, s, err, g.C);
    case 3: return launch_g<3>(a, s, err, g.C);
    default: return launch_g<4>(a, s, err, g.C);
  }
}

}  // namespace dsa
