// Exact Top-K over scores spread across the CTAs of one thread-block cluster.
//
// "Deep Dive into Sparse Attention and Engineering Optimizations for Efficient Inference
// in Kimi K3.1 Pro", section 2.1: selection happens on chip, with no intermediate score
// write-back.  Each CTA of the cluster holds the order-preserving keys of one contiguous
// chunk of positions in shared memory (key 0 = not selectable).  The K-th largest key T
// is found by a three-digit radix select (11 + 11 + 10 bits) whose histograms are summed
// in the leader CTA's shared memory through distributed shared memory; then every CTA
// writes its positions with key > T, and the lowest positions with key == T up to K
// (CTA rank order is position order, so the tie quota is handed out rank by rank).
#pragma once

#include "dsa_common.cuh"

namespace dsa {

constexpr int kHistBins = 2048;

// Shared-memory scratch of the selector (one per CTA; the leader's copy is the
// cluster-wide one).
struct TopkSmem {
  uint32_t hist[2][kHistBins];   // leader: cluster histograms (double-buffered)
  uint32_t local[kHistBins];     // every CTA: its own histogram
  uint32_t counts[2][16];        // leader: per-rank (count_gt, count_eq)
  uint32_t bcast[2];             // every CTA: (digit, count_above) sent by the leader
  uint32_t warp_tot[2][32];      // block scan scratch
};

// Zero the leader's histograms; call before the first cluster_sync of the kernel.
__device__ __forceinline__ void topk_init(TopkSmem& sm) {
  for (int i = threadIdx.x; i < 2 * kHistBins; i += blockDim.x) (&sm.hist[0][0])[i] = 0;
}

// Block-wide exclusive scan of two 0/1 flags; returns the exclusive prefix of each and
// writes the block totals.
__device__ __forceinline__ void block_scan2(TopkSmem& sm, uint32_t f0, uint32_t f1, uint32_t& p0,
                                            uint32_t& p1, uint32_t& t0, uint32_t& t1) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const uint32_t b0 = __ballot_sync(0xffffffffu, f0), b1 = __ballot_sync(0xffffffffu, f1);
  const uint32_t lt = (1u << lane) - 1u;
  if (lane == 0) { sm.warp_tot[0][warp] = __popc(b0); sm.warp_tot[1][warp] = __popc(b1); }
  __syncthreads();
  uint32_t o0 = 0, o1 = 0, s0 = 0, s1 = 0;
  for (int i = 0; i < nw; ++i) {
    const uint32_t a = sm.warp_tot[0][i], b = sm.warp_tot[1][i];
    if (i < warp) { o0 += a; o1 += b; }
    s0 += a; s1 += b;
  }
  p0 = o0 + __popc(b0 & lt);
  p1 = o1 + __popc(b1 & lt);
  t0 = s0; t1 = s1;
  __syncthreads();
}

// Select the Top-K of one query row.
//   keys[0..len)  this CTA's keys for positions c0 .. c0+len-1 (0 = not selectable)
//   n_sel         number of selectable positions of the row (positions 0..n_sel-1)
// Writes out_idx[0..K) (and out_scores if non-null).  Must be called by every thread of
// every CTA of the cluster (it contains cluster barriers).
__device__ void cluster_topk_row(TopkSmem& sm, const uint32_t* keys, int c0, int len, int n_sel,
                                 int K, int32_t* out_idx, float* out_scores) {
  const uint32_t rank = cluster_ctarank();
  const uint32_t nrank = cluster_nctarank();
  const int tid = threadIdx.x, nt = blockDim.x;

  if (n_sel <= K) {
    // every selectable position is kept, in position order; rank 0 pads the tail
    for (int i = tid; i < len; i += nt) {
      const int p = c0 + i;
      if (p < n_sel) {
        out_idx[p] = p;
        if (out_scores) out_scores[p] = key_score(keys[i]);
      }
    }
    if (rank == 0) {
      for (int s = n_sel + tid; s < K; s += nt) {
        out_idx[s] = -1;
        if (out_scores) out_scores[s] = -INFINITY;
      }
    }
    return;
  }

  uint32_t prefix = 0;
  uint32_t need = static_cast<uint32_t>(K);
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
#pragma unroll 1
  for (int lvl = 0; lvl < 3; ++lvl) {
    const int sh = shifts[lvl];
    const uint32_t mask = (1u << widths[lvl]) - 1u;
    const int hsh = sh + widths[lvl];  // bits above this digit must equal prefix's
    uint32_t* cl_hist = sm.hist[lvl & 1];
    for (int i = tid; i < kHistBins; i += nt) sm.local[i] = 0;
    __syncthreads();
    for (int base = 0; base < len; base += nt) {  // uniform trip count: whole warps
      const int i = base + tid;
      const uint32_t k = (i < len) ? keys[i] : 0u;
      const bool hit = (k != 0u) && (hsh >= 32 || (k >> hsh) == (prefix >> hsh));
      const uint32_t d = hit ? ((k >> sh) & mask) : 0xFFFFFFFFu;
      // warp-aggregated shared atomics: scores crowd into a few top-digit bins
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      if (hit && (__ffs(peers) - 1) == (tid & 31)) atomicAdd(&sm.local[d], __popc(peers));
    }
    __syncthreads();
    for (int i = tid; i < kHistBins; i += nt) {
      const uint32_t c = sm.local[i];
      if (c) dsmem_add_u32(dsmem_addr(&cl_hist[i], 0), c);
    }
    cluster_sync();
    if (rank == 0) {
      // find digit d (scanning from the top) where the running count reaches `need`
      if (tid < 32) {
        uint32_t run = 0, found_d = 0, found_above = 0;
        bool found = false;
        const int per = kHistBins / 32;  // each lane sums one 64-bin slice (top slice first)
        const int lane = tid;
        const int hi = kHistBins - lane * per;  // slice [hi - per, hi)
        uint32_t slice = 0;
        for (int j = hi - per; j < hi; ++j) slice += cl_hist[j];
        // inclusive prefix over lanes (lane 0 = top slice)
        uint32_t incl = slice;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const uint32_t excl = incl - slice;
        const bool mine = (excl < need) && (need <= incl);
        const uint32_t who = __ballot_sync(0xffffffffu, mine);
        const int src = __ffs(who) - 1;
        if (lane == src) {
          run = excl;
          for (int j = hi - 1; j >= hi - per; --j) {
            const uint32_t c = cl_hist[j];
            if (!found && run + c >= need) { found = true; found_d = j; found_above = run; }
            run += c;
          }
          for (uint32_t r = 0; r < nrank; ++r) {
            dsmem_st_u32(dsmem_addr(&sm.bcast[0], r), found_d);
            dsmem_st_u32(dsmem_addr(&sm.bcast[1], r), found_above);
          }
        }
      }
      __syncthreads();
      for (int i = tid; i < kHistBins; i += nt) cl_hist[i] = 0;  // ready for reuse
    }
    cluster_sync();
    prefix |= sm.bcast[0] << sh;
    need -= sm.bcast[1];
  }
  const uint32_t T = prefix;
  const uint32_t need_eq = need;  // >= 1

  // count > T and == T locally, publish to the leader
  uint32_t n_gt = 0, n_eq = 0;
  for (int i = tid; i < len; i += nt) {
    const uint32_t k = keys[i];
    n_gt += (k > T);
    n_eq += (k == T);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    n_gt += __shfl_xor_sync(0xffffffffu, n_gt, o);
    n_eq += __shfl_xor_sync(0xffffffffu, n_eq, o);
  }
  if ((tid & 31) == 0) { sm.warp_tot[0][tid >> 5] = n_gt; sm.warp_tot[1][tid >> 5] = n_eq; }
  __syncthreads();
  if (tid == 0) {
    uint32_t a = 0, b = 0;
    for (int i = 0; i < (nt >> 5); ++i) { a += sm.warp_tot[0][i]; b += sm.warp_tot[1][i]; }
    dsmem_st_u32(dsmem_addr(&sm.counts[0][rank], 0), a);
    dsmem_st_u32(dsmem_addr(&sm.counts[1][rank], 0), b);
  }
  cluster_sync();
  uint32_t gt_before = 0, eq_before = 0, gt_total = 0;
  for (uint32_t r = 0; r < nrank; ++r) {
    const uint32_t a = dsmem_ld_u32(dsmem_addr(&sm.counts[0][r], 0));
    const uint32_t b = dsmem_ld_u32(dsmem_addr(&sm.counts[1][r], 0));
    if (r < rank) { gt_before += a; eq_before += b; }
    gt_total += a;
  }
  const uint32_t eq_take_lo = eq_before < need_eq ? eq_before : need_eq;  // first eq slot
  uint32_t gt_off = gt_before;
  uint32_t eq_off = gt_total + eq_take_lo;
  uint32_t eq_left = need_eq - eq_take_lo;  // tie quota still open for this rank onwards

  // ordered compaction over the chunk (ties must go to the lowest positions)
  for (int base = 0; base < len; base += nt) {
    const int i = base + tid;
    const uint32_t k = (i < len) ? keys[i] : 0u;
    const uint32_t fg = (k > T), fe = (k == T) && (k != 0u);
    uint32_t pg, pe, tg, te;
    block_scan2(sm, fg, fe, pg, pe, tg, te);
    // (the slot bounds only guard the row against an inconsistent count; they never bind)
    if (fg && gt_off + pg < static_cast<uint32_t>(K)) {
      out_idx[gt_off + pg] = c0 + i;
      if (out_scores) out_scores[gt_off + pg] = key_score(k);
    }
    if (fe && pe < eq_left && eq_off + pe < static_cast<uint32_t>(K)) {
      out_idx[eq_off + pe] = c0 + i;
      if (out_scores) out_scores[eq_off + pe] = key_score(k);
    }
    gt_off += tg;
    const uint32_t used = te < eq_left ? te : eq_left;
    eq_off += used;
    eq_left -= used;
  }
  // keep the leader's counts alive until every rank has read them
  cluster_sync();
}

}  // namespace dsa
