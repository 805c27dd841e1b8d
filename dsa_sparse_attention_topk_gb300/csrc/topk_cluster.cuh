// Exact Top-K over scores spread across the CTAs of one thread-block cluster.
//
// "Deep Dive into Sparse Attention and Engineering Optimizations for Efficient Inference
// in Kimi K3.1 Pro", section 2.1: selection happens on chip, with no intermediate score
// write-back.  Each CTA of the cluster holds the order-preserving keys of one contiguous
// chunk of positions in shared memory (key 0 = not selectable).  The K-th largest key T
// is found by a three-digit radix select (11 + 11 + 10 bits) whose histograms are summed
// in the leader CTA's shared memory through distributed shared memory.  The first
// digit's local histogram is built while the scores are produced; the later digits only
// touch keys that share the selected prefix.  Every CTA then writes its positions with
// key > T, and the lowest positions with key == T up to K (CTA rank order is position
// order, so the tie quota is handed out rank by rank).  The output of every CTA is in
// position order, so the result is deterministic.
#pragma once

#include "dsa_common.cuh"

namespace dsa {

constexpr int kHistBins = 2048;

// Shared-memory scratch of the selector (one per CTA; the leader's copy is the
// cluster-wide one).
struct TopkSmem {
  uint32_t hist[2][kHistBins];   // leader: cluster histograms (double-buffered)
  uint32_t local[kHistBins];     // every CTA: its histogram of the current digit
  uint32_t counts[2][16];        // every CTA: per-rank (count_gt, count_eq), pushed by each rank
  uint32_t bcast[2];             // every CTA: (digit, count_above) sent by the leader
  uint32_t warp_cnt[2][32];      // per-warp counts for the ordered compaction
};

// Zero the leader's histograms; call before the first cluster_sync of the kernel.
__device__ __forceinline__ void topk_init(TopkSmem& sm) {
  for (int i = threadIdx.x; i < 2 * kHistBins; i += blockDim.x) (&sm.hist[0][0])[i] = 0;
}

// Add `key`'s top digit (bits 31..21) to a local histogram, aggregated over the warp.
// Every lane of the warp must call it (key 0 = nothing to add).
__device__ __forceinline__ void hist_add_top_digit(uint32_t* hist, uint32_t key) {
  const uint32_t d = key ? (key >> 21) : 0xFFFFFFFFu;
  const uint32_t peers = __match_any_sync(0xffffffffu, d);
  if (key && (__ffs(peers) - 1) == static_cast<int>(threadIdx.x & 31)) atomicAdd(&hist[d], __popc(peers));
}

// Leader: find the digit (scanning down from the top bin) where the running count of
// cl_hist reaches `need`, send (digit, count above it) to every rank, zero cl_hist.
// One warp: each lane sums a 64-bin slice (lane 0 = the top slice), a shuffle scan finds
// the slice that crosses `need`, and the warp scans that slice two bins per lane.
__device__ __forceinline__ void leader_pick(TopkSmem& sm, uint32_t* cl_hist, uint32_t need, uint32_t nrank) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    constexpr int per = kHistBins / 32;
    const int lane = tid;
    const int hi = kHistBins - lane * per;  // lane's slice [hi - per, hi)
    const uint4* h4 = reinterpret_cast<const uint4*>(cl_hist + hi - per);
    uint32_t slice = 0;
#pragma unroll
    for (int j = 0; j < per / 4; ++j) {
      const uint4 v = h4[j];
      slice += (v.x + v.y) + (v.z + v.w);
    }
    uint32_t incl = slice;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const uint32_t excl = incl - slice;
    const uint32_t who = __ballot_sync(0xffffffffu, (excl < need) && (need <= incl));
    const int src = __ffs(who) - 1;  // the slice holding the crossing (always found)
    const uint32_t base = __shfl_sync(0xffffffffu, excl, src < 0 ? 0 : src);
    const int top = kHistBins - (src < 0 ? 0 : src) * per;
    // bins of that slice in descending order: lane l holds top-1-2l and top-2-2l
    const uint32_t c0 = cl_hist[top - 1 - 2 * lane], c1 = cl_hist[top - 2 - 2 * lane];
    const uint32_t pair = c0 + c1;
    uint32_t pin = pair;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, pin, o);
      if (lane >= o) pin += v;
    }
    const uint32_t above0 = base + pin - pair;          // count above bin top-1-2l
    const bool hit0 = above0 < need && need <= above0 + c0;
    const bool hit1 = !hit0 && above0 + c0 < need && need <= above0 + pair;
    const uint32_t found = __ballot_sync(0xffffffffu, hit0 || hit1);
    if (src >= 0 && lane == __ffs(found) - 1) {
      const uint32_t found_d = hit0 ? static_cast<uint32_t>(top - 1 - 2 * lane) : static_cast<uint32_t>(top - 2 - 2 * lane);
      const uint32_t found_above = hit0 ? above0 : above0 + c0;
      for (uint32_t r = 0; r < nrank; ++r) {
        dsmem_st_u32(dsmem_addr(&sm.bcast[0], r), found_d);
        dsmem_st_u32(dsmem_addr(&sm.bcast[1], r), found_above);
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < kHistBins; i += blockDim.x) cl_hist[i] = 0;  // ready for reuse
}

// Select the Top-K of one query row.
//   keys[0..len)  this CTA's keys for positions c0 .. c0+len-1 (0 = not selectable)
//   hist0         this CTA's histogram of the keys' top digit (bits 31..21); it is
//                 consumed (left in an unspecified state)
//   n_sel         number of selectable positions of the row (positions 0..n_sel-1)
// Writes out_idx[0..K) (and out_scores if non-null).  Must be called by every thread of
// every CTA of the cluster (it contains cluster barriers).
__device__ void cluster_topk_row(TopkSmem& sm, const uint32_t* keys, uint32_t* hist0, int c0, int len, int n_sel,
                                 int K, int32_t* out_idx, float* out_scores) {
  const uint32_t rank = cluster_ctarank();
  const uint32_t nrank = cluster_nctarank();
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;

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
#pragma unroll 1
  for (int lvl = 0; lvl < 3; ++lvl) {
    const int sh = lvl == 0 ? 21 : (lvl == 1 ? 10 : 0);
    const int width = lvl == 2 ? 10 : 11;
    const uint32_t mask = (1u << width) - 1u;
    const int hsh = sh + width;  // bits above this digit must equal prefix's
    uint32_t* lh = lvl == 0 ? hist0 : sm.local;
    uint32_t* cl_hist = sm.hist[lvl & 1];
    if (lvl > 0) {
      for (int i = tid; i < kHistBins; i += nt) sm.local[i] = 0;
      __syncthreads();
      for (int i = tid; i < len; i += nt) {
        const uint32_t k = keys[i];
        if (k != 0u && (k >> hsh) == (prefix >> hsh)) atomicAdd(&sm.local[(k >> sh) & mask], 1u);
      }
    }
    __syncthreads();
    for (int i = tid; i < kHistBins; i += nt) {
      const uint32_t c = lh[i];
      if (c) dsmem_add_u32(dsmem_addr(&cl_hist[i], 0), c);
    }
    cluster_sync();
    if (rank == 0) leader_pick(sm, cl_hist, need, nrank);
    cluster_sync();
    prefix |= sm.bcast[0] << sh;
    need -= sm.bcast[1];
  }
  const uint32_t T = prefix;
  const uint32_t need_eq = need;  // >= 1

  // counts of this CTA's keys above and at T, per warp (warp w owns the contiguous slice
  // [w*span, (w+1)*span) of the chunk), then per CTA through the leader
  const int span = ((len + nw - 1) / nw + 31) / 32 * 32;
  const int lo = warp * span, hi = min(len, lo + span);
  uint32_t cg = 0, ce = 0;
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const uint32_t k = i < hi ? keys[i] : 0u;
    cg += __popc(__ballot_sync(0xffffffffu, k > T));
    ce += __popc(__ballot_sync(0xffffffffu, k == T && k != 0u));
  }
  if (lane == 0) { sm.warp_cnt[0][warp] = cg; sm.warp_cnt[1][warp] = ce; }
  __syncthreads();
  if (tid < static_cast<int>(nrank)) {  // push this rank's counts into every rank's table
    uint32_t my_gt = 0, my_eq = 0;
    for (int w = 0; w < nw; ++w) { my_gt += sm.warp_cnt[0][w]; my_eq += sm.warp_cnt[1][w]; }
    dsmem_st_u32(dsmem_addr(&sm.counts[0][rank], tid), my_gt);
    dsmem_st_u32(dsmem_addr(&sm.counts[1][rank], tid), my_eq);
  }
  cluster_sync();
  uint32_t gt_before = 0, eq_before = 0, gt_total = 0;
  for (uint32_t r = 0; r < nrank; ++r) {
    const uint32_t a = sm.counts[0][r], b = sm.counts[1][r];
    if (r < rank) { gt_before += a; eq_before += b; }
    gt_total += a;
  }
  const uint32_t eq_lo = eq_before < need_eq ? eq_before : need_eq;
  const uint32_t eq_quota = need_eq - eq_lo;  // ties this CTA may still take

  // ordered compaction of each warp's slice
  uint32_t og = gt_before, oe = 0;
  for (int w = 0; w < warp; ++w) { og += sm.warp_cnt[0][w]; oe += sm.warp_cnt[1][w]; }
  const uint32_t lt = (1u << lane) - 1u;
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const uint32_t k = i < hi ? keys[i] : 0u;
    const uint32_t bg = __ballot_sync(0xffffffffu, k > T);
    const uint32_t be = __ballot_sync(0xffffffffu, k == T && k != 0u);
    if (k > T) {
      const uint32_t slot = og + __popc(bg & lt);
      if (slot < static_cast<uint32_t>(K)) {  // guards the row against an inconsistent count
        out_idx[slot] = c0 + i;
        if (out_scores) out_scores[slot] = key_score(k);
      }
    }
    if (k == T && k != 0u) {
      const uint32_t r = oe + __popc(be & lt);
      if (r < eq_quota) {
        const uint32_t slot = gt_total + eq_lo + r;
        if (slot < static_cast<uint32_t>(K)) {
          out_idx[slot] = c0 + i;
          if (out_scores) out_scores[slot] = key_score(k);
        }
      }
    }
    og += __popc(bg);
    oe += __popc(be);
  }
  // keep the leader's counts alive until every rank has read them
  cluster_sync();
}

}  // namespace dsa
