// Exact Top-K over scores spread across the CTAs of one thread-block cluster.
//
// "Deep Dive into Sparse Attention and Engineering Optimizations for Efficient Inference
// in Kimi K3.1 Pro", section 2.1: selection happens on chip, with no intermediate score
// write-back.  Each CTA of the cluster holds the order-preserving keys of one contiguous
// chunk of positions in shared memory (key 0 = not selectable).  The K-th largest key T
// is found by a three-digit radix select (11 + 11 + 10 bits).
//
// First digit: each CTA builds the histogram of its keys' top 11 bits while the scores are
// produced, adds it into every CTA's copy over distributed shared memory, and after one
// cluster barrier every CTA picks the digit d0 holding the K-th key on its own.
//
// Then, when the keys of bin d0 fit in one CTA's (now idle) copy ring, every CTA counts its
// keys above bin d0 and in it, and the counts are exchanged (second barrier).  Each CTA
// writes its keys above d0 straight to the output at its rank's offset, and its keys in
// bin d0 with their positions into the leader's list at its rank's offset, both in
// position order.  The list entries are asynchronous stores that the leader's mbarrier
// counts (it expects the bin's cluster-wide count), so neither the list nor the output
// writes wait on a cluster barrier.  The leader finishes alone over those few candidates:
// the last two digits, then the keys > T and the lowest positions with key == T.
//
// Otherwise (a top bin too crowded for the list) the last two digits go through the
// cluster as well: their histograms are summed in the leader, which broadcasts each digit,
// and every CTA writes its own keys > T and its share of the ties (CTA rank order is
// position order, so the tie quota is handed out rank by rank).
//
// Either way the output is deterministic.
#pragma once

#include <cstddef>

#include "dsa_common.cuh"
#include "tc_utils.cuh"

namespace dsa {

constexpr int kHistBins = 2048;

// Shared-memory scratch of the selector (one per CTA).
struct TopkSmem {
  uint32_t hist[2][kHistBins];   // [0]: the cluster's first-digit histogram (every CTA);
                                 // leader: cluster histograms of the later digits
  uint32_t local[kHistBins];     // this CTA's histogram of the current digit
  uint32_t counts[2][2][16];     // per-rank counts, one table per row parity
  uint32_t bcast[2];             // (digit, count_above) sent by the leader
  uint32_t pick[4];              // results of this CTA's own picks
  uint32_t warp_cnt[2][32];      // per-warp counts for the ordered compactions
  uint32_t few[32];              // leader: the candidates that share T's top 22 bits
  uint32_t n_few;                // leader: how many there are (only the first 32 are kept)
  uint32_t cand_uses;            // leader: rows whose candidates came through cand_bar
  uint64_t cand_bar;             // leader: completes once a row's candidates have landed
};
static_assert(offsetof(TopkSmem, hist) % 16 == 0 && offsetof(TopkSmem, local) % 16 == 0,
              "the histograms are accessed 16 bytes at a time");

// Zero the histograms and set up the candidate barrier; call with every thread before the
// cluster barrier that precedes any DSMEM traffic.
__device__ __forceinline__ void topk_init(TopkSmem& sm) {
  for (int i = threadIdx.x; i < 2 * kHistBins; i += blockDim.x) (&sm.hist[0][0])[i] = 0;
  if (threadIdx.x == 0) {
    sm.cand_uses = 0;
    tc::mbar_init(&sm.cand_bar, 1);
    tc::mbar_fence_init();
  }
}

// Add `key`'s top digit (bits 31..21) to a local histogram, aggregated over the warp.
// Every lane of the warp must call it (key 0 = nothing to add).
__device__ __forceinline__ void hist_add_top_digit(uint32_t* hist, uint32_t key) {
  const uint32_t d = key ? (key >> 21) : 0xFFFFFFFFu;
  const uint32_t peers = __match_any_sync(0xffffffffu, d);
  if (key && (__ffs(peers) - 1) == static_cast<int>(threadIdx.x & 31)) atomicAdd(&hist[d], __popc(peers));
}

// One warp (all 32 lanes): the digit d where the running count of `hist`, scanned down
// from the top bin, reaches `need`, and the count of the bins above d.  Each lane sums a
// 64-bin slice (lane 0 = the top slice), a shuffle scan finds the slice that crosses
// `need`, and the warp scans that slice two bins per lane.  Every lane gets the result;
// false (and d = above = 0) if the histogram holds fewer than `need`.
// Not inlined: its call sites run once each, so one shared copy stays warm in the
// instruction cache.
__device__ __noinline__ uint3 warp_pick_impl(const uint32_t* hist, uint32_t need) {
  constexpr int per = kHistBins / 32;
  const int lane = threadIdx.x & 31;
  const int hi = kHistBins - lane * per;  // lane's slice [hi - per, hi)
  const uint4* h4 = reinterpret_cast<const uint4*>(hist + hi - per);
  uint32_t slice = 0;
  // lane l starts l vectors into its slice: the warp's 32 loads of each step then spread
  // over the banks (slices are 256 bytes apart, so a common order would conflict 32-way)
#pragma unroll
  for (int j = 0; j < per / 4; ++j) {
    const uint4 v = h4[(j + lane) & (per / 4 - 1)];
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
  if (!who) return make_uint3(0u, 0u, 0u);
  const int src = __ffs(who) - 1;
  const uint32_t base = __shfl_sync(0xffffffffu, excl, src);
  const int top = kHistBins - src * per;
  // bins of that slice in descending order: lane l holds top-1-2l and top-2-2l
  const uint32_t c0 = hist[top - 1 - 2 * lane], c1 = hist[top - 2 - 2 * lane];
  const uint32_t pair = c0 + c1;
  uint32_t pin = pair;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, pin, o);
    if (lane >= o) pin += v;
  }
  const uint32_t above0 = base + pin - pair;  // count above bin top-1-2l
  const bool hit0 = above0 < need && need <= above0 + c0;
  const bool hit1 = !hit0 && above0 + c0 < need && need <= above0 + pair;
  const uint32_t found = __ballot_sync(0xffffffffu, hit0 || hit1);
  if (!found) return make_uint3(0u, 0u, 0u);
  const int fl = __ffs(found) - 1;
  const uint32_t d = hit0 ? static_cast<uint32_t>(top - 1 - 2 * lane) : static_cast<uint32_t>(top - 2 - 2 * lane);
  const uint32_t ab = hit0 ? above0 : above0 + c0;
  return make_uint3(__shfl_sync(0xffffffffu, d, fl), __shfl_sync(0xffffffffu, ab, fl), 1u);
}
// (the result comes back in registers: reference out-parameters would put the caller's
// variables in local memory, whose first touch after the scan misses L1)
__device__ __forceinline__ bool warp_pick(const uint32_t* hist, uint32_t need, uint32_t& digit, uint32_t& above) {
  const uint3 r = warp_pick_impl(hist, need);
  digit = r.x;
  above = r.y;
  return r.z != 0;
}

// Leader: pick on the cluster histogram cl_hist, send (digit, count above it) to every
// rank, zero cl_hist.
__device__ __forceinline__ void leader_pick(TopkSmem& sm, uint32_t* cl_hist, uint32_t need, uint32_t nrank) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    uint32_t d, ab;
    warp_pick(cl_hist, need, d, ab);
    if (tid == 0) {
      for (uint32_t r = 0; r < nrank; ++r) {
        dsmem_st_u32(dsmem_addr(&sm.bcast[0], r), d);
        dsmem_st_u32(dsmem_addr(&sm.bcast[1], r), ab);
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < kHistBins; i += blockDim.x) cl_hist[i] = 0;  // ready for reuse
}

// Block-local pick on this CTA's histogram: (digit, count above) for every thread.
__device__ __forceinline__ void block_pick(TopkSmem& sm, const uint32_t* hist, uint32_t need, uint32_t& d,
                                           uint32_t& above) {
  if (threadIdx.x < 32) {
    uint32_t dd, ab;
    const bool found = warp_pick(hist, need, dd, ab);
    if (threadIdx.x == 0) { sm.pick[0] = dd; sm.pick[1] = ab; sm.pick[2] = found ? 1u : 0u; sm.pick[3] = hist[dd]; }
  }
  __syncthreads();
  d = sm.pick[0];
  above = sm.pick[1];
}

// Warp w of the block owns the contiguous slice [w*span, (w+1)*span) of n items; span is
// a multiple of `unit` items.
__device__ __forceinline__ int warp_span(int n, int unit = 32) {
  const int nw = blockDim.x >> 5;
  return ((n + nw - 1) / nw + unit - 1) / unit * unit;
}

// Leader, after the barrier that publishes the candidates: cand[0..n) holds, in position
// order, every key whose top digit is d0 (the bin of the K-th key); above0 keys lie above
// that bin and are already written.  Finish the last two digits over the candidates and
// write the selected ones after them: keys > T in position order, then the lowest
// positions with key == T.
// The caller zeroes sm.local and sm.n_few and passes a block barrier first.
__device__ void leader_finish(TopkSmem& sm, const uint2* cand, uint32_t n, uint32_t d0, uint32_t above0, int K,
                              int32_t* out_idx, float* out_scores) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  uint32_t need = static_cast<uint32_t>(K) - above0;
  for (uint32_t v = tid; v < n; v += nt) atomicAdd(&sm.local[(cand[v].x >> 10) & 2047u], 1u);
  __syncthreads();
  uint32_t d1, a1;
  block_pick(sm, sm.local, need, d1, a1);
  need -= a1;
  const uint32_t pre = (d0 << 11) | d1;  // bits 31..10 of T
  // Last digit.  The candidates that share T's top 22 bits are usually a handful: they are
  // collected, and one warp finds T as the need-th largest of them (the largest key that
  // at least `need` of them reach).  More than 32 take a histogram of the last 10 bits.
  for (int i = tid; i < kHistBins; i += nt) sm.local[i] = 0;
  for (uint32_t v = tid; v < n; v += nt) {
    const uint32_t k = cand[v].x;
    if ((k >> 10) == pre) {
      const uint32_t slot = atomicAdd(&sm.n_few, 1u);
      if (slot < 32u) sm.few[slot] = k;
    }
  }
  __syncthreads();
  uint32_t T = 0u, a2 = 0u;
  bool found = false;
  if (sm.n_few <= 32u) {
    if (warp == 0) {
      const uint32_t nf = sm.n_few;
      const uint32_t key = static_cast<uint32_t>(lane) < nf ? sm.few[lane] : 0u;
      uint32_t ge = 0;  // how many of them are >= this lane's key
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t kj = __shfl_sync(0xffffffffu, key, j);
        ge += (static_cast<uint32_t>(j) < nf && kj >= key) ? 1u : 0u;
      }
      const bool q = static_cast<uint32_t>(lane) < nf && ge >= need;
      const uint32_t t = __reduce_max_sync(0xffffffffu, q ? key : 0u);
      const uint32_t above = __reduce_add_sync(0xffffffffu, (static_cast<uint32_t>(lane) < nf && key > t) ? 1u : 0u);
      const bool ok = __any_sync(0xffffffffu, q);
      if (lane == 0) { sm.pick[0] = t; sm.pick[1] = above; sm.pick[2] = ok ? 1u : 0u; }
    }
    __syncthreads();
    found = sm.pick[2] != 0u;
    T = sm.pick[0];
    a2 = sm.pick[1];
    __syncthreads();  // every thread has read the picks before they are written again
  }
  if (!found) {
    for (uint32_t v = tid; v < n; v += nt) {
      const uint32_t k = cand[v].x;
      if ((k >> 10) == pre) atomicAdd(&sm.local[k & 1023u], 1u);
    }
    __syncthreads();
    uint32_t d2;
    block_pick(sm, sm.local, need, d2, a2);
    T = (pre << 10) | d2;
  }
  const uint32_t need_eq = need - a2;                     // >= 1
  const uint32_t gt_total = static_cast<uint32_t>(K) - need_eq;

  // one ordered pass over the candidates: keys > T after the above0 ones, then the first
  // need_eq keys == T
  const int span = warp_span(static_cast<int>(n));
  const int lo = warp * span, hi = min(static_cast<int>(n), lo + span);
  uint32_t cg = 0, ce = 0;
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const uint32_t k = i < hi ? cand[i].x : 0u;
    cg += __popc(__ballot_sync(0xffffffffu, k > T));
    ce += __popc(__ballot_sync(0xffffffffu, k == T && k != 0u));
  }
  if (lane == 0) { sm.warp_cnt[0][warp] = cg; sm.warp_cnt[1][warp] = ce; }
  __syncthreads();
  uint32_t og = above0, oe = 0;
  for (int w = 0; w < warp; ++w) { og += sm.warp_cnt[0][w]; oe += sm.warp_cnt[1][w]; }
  const uint32_t lt = (1u << lane) - 1u;
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const uint2 e = i < hi ? cand[i] : make_uint2(0u, 0u);
    const uint32_t k = e.x;
    const uint32_t bg = __ballot_sync(0xffffffffu, k > T);
    const uint32_t be = __ballot_sync(0xffffffffu, k == T && k != 0u);
    uint32_t slot = 0xFFFFFFFFu;
    if (k > T) slot = og + __popc(bg & lt);
    if (k == T && k != 0u) {
      const uint32_t r = oe + __popc(be & lt);
      if (r < need_eq) slot = gt_total + r;
    }
    if (slot < static_cast<uint32_t>(K)) {  // guards the row against an inconsistent count
      out_idx[slot] = static_cast<int32_t>(e.y);
      if (out_scores) out_scores[slot] = key_score(k);
    }
    og += __popc(bg);
    oe += __popc(be);
  }
}

// Every CTA writes its keys > T (in position order, after the lower ranks') and its share
// of the first need_eq keys == T (rank order is position order) to the output; returns the
// cluster-wide count of keys > T.  Called by every thread of every CTA of the cluster.
__device__ uint32_t cluster_write_selected(TopkSmem& sm, const uint32_t* keys, int c0, int len, uint32_t T,
                                          uint32_t need_eq, int K, int32_t* out_idx, float* out_scores, int par) {
  const uint32_t rank = cluster_ctarank();
  const uint32_t nrank = cluster_nctarank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  // counts of this CTA's keys above and at T, per warp, then per CTA through every rank
  const int span = warp_span(len);
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
    dsmem_st_u32(dsmem_addr(&sm.counts[par][0][rank], tid), my_gt);
    dsmem_st_u32(dsmem_addr(&sm.counts[par][1][rank], tid), my_eq);
  }
  cluster_sync();
  uint32_t gt_before = 0, eq_before = 0, gt_total = 0;
  for (uint32_t r = 0; r < nrank; ++r) {
    const uint32_t a = sm.counts[par][0][r], b = sm.counts[par][1][r];
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
  // keep the counts alive until every rank has read them
  cluster_sync();
  return gt_total;
}

// Select the Top-K of one query row.
//   keys[0..len)  this CTA's keys for positions c0 .. c0+len-1 (0 = not selectable);
//                 16-byte aligned; chunk >= len is the chunk size of every CTA
//   hist0         this CTA's histogram of the keys' top digit (bits 31..21); read only
//   n_sel         number of selectable positions of the row (positions 0..n_sel-1)
//   cand          cand_cap free (key, position) slots of shared memory, at the same offset
//                 in every CTA of the cluster (the leader's copy receives the candidates)
//   row           index of this call among the kernel's calls (its parity picks the count
//                 table, so a CTA that runs ahead never overwrites counts still being read)
//   status, wait_ns  the leader's wait for the candidates gives up after wait_ns and sets
//                 the TIMEOUT status bit
// Writes out_idx[0..K) (and out_scores if non-null).  Must be called by every thread of
// every CTA of the cluster (it contains cluster barriers).  The caller must pass another
// cluster barrier before `cand` or the selector's scratch is written again.
__device__ void cluster_topk_row(TopkSmem& sm, const uint32_t* keys, const uint32_t* hist0, int c0, int chunk, int len,
                                 int n_sel, int K, int32_t* out_idx, float* out_scores, uint2* cand, int cand_cap,
                                 int row, unsigned* status, uint64_t wait_ns) {
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

  // ---- first digit: every CTA sums all ranks' histograms (final since the caller's
  // cluster barrier, and never written again) into its own copy and picks locally ----
  for (int i = 4 * tid; i < kHistBins; i += 4 * nt) {
    uint4 sum = *reinterpret_cast<const uint4*>(hist0 + i);
    for (uint32_t r = 0; r < nrank; ++r) {
      if (r == rank) continue;
      const uint4 v = dsmem_ld_v4(dsmem_addr(hist0 + i, r));
      sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
    }
    *reinterpret_cast<uint4*>(&sm.hist[0][i]) = sum;
  }
  __syncthreads();
  uint32_t d0, above0;
  block_pick(sm, sm.hist[0], static_cast<uint32_t>(K), d0, above0);
  const bool found = sm.pick[2] != 0;
  // every thread has read the picks; the copy is refilled only after a later cluster barrier
  for (int i = tid; i < kHistBins; i += nt) sm.hist[0][i] = 0;
  if (!found) {
    // fewer than K selectable keys although n_sel > K (positions on pages flagged bad):
    // keep every selectable key, in position order, and pad the rest of the row with -1
    const uint32_t n_valid = cluster_write_selected(sm, keys, c0, len, 0u, 0u, K, out_idx, out_scores, row & 1);
    if (rank == 0) {
      for (int s = static_cast<int>(n_valid) + tid; s < K; s += nt) {
        out_idx[s] = -1;
        if (out_scores) out_scores[s] = -INFINITY;
      }
    }
    return;
  }

  const uint32_t at_total = sm.pick[3];  // cluster-wide count of keys in bin d0
  if (at_total <= static_cast<uint32_t>(cand_cap)) {
    const int par = row & 1;
    // the leader's barrier expects at_total candidates of 8 bytes; they arrive only after
    // the counts barrier below, so the expectation is in place first
    const uint32_t cand_parity = sm.cand_uses & 1u;
    if (rank == 0 && tid == 0) tc::mbar_arrive_expect_tx(&sm.cand_bar, at_total * static_cast<uint32_t>(sizeof(uint2)));
    // ---- (1) this CTA's keys above bin d0 and in it, counted per warp slice ----
    const int span = warp_span(len);
    const int lo = warp * span, hi = min(len, lo + span);
    uint32_t cg = 0, ce = 0;
    for (int base = lo; base < hi; base += 32) {
      const int i = base + lane;
      const uint32_t k = i < hi ? keys[i] : 0u;
      const uint32_t dg = k >> 21;
      cg += __popc(__ballot_sync(0xffffffffu, k != 0u && dg > d0));
      ce += __popc(__ballot_sync(0xffffffffu, k != 0u && dg == d0));
    }
    if (lane == 0) { sm.warp_cnt[0][warp] = cg; sm.warp_cnt[1][warp] = ce; }
    __syncthreads();
    if (tid < static_cast<int>(nrank)) {  // push this rank's totals into every rank's table
      uint32_t my_gt = 0, my_eq = 0;
      for (int w = 0; w < nw; ++w) { my_gt += sm.warp_cnt[0][w]; my_eq += sm.warp_cnt[1][w]; }
      dsmem_st_u32(dsmem_addr(&sm.counts[par][0][rank], tid), my_gt);
      dsmem_st_u32(dsmem_addr(&sm.counts[par][1][rank], tid), my_eq);
    }
    cluster_sync();  // every rank's totals are known everywhere
    uint32_t og = 0, oe = 0;  // this warp's first output slot / candidate slot
    for (uint32_t r = 0; r < rank; ++r) { og += sm.counts[par][0][r]; oe += sm.counts[par][1][r]; }
    for (int w = 0; w < warp; ++w) { og += sm.warp_cnt[0][w]; oe += sm.warp_cnt[1][w]; }
    // ---- (2) keys above bin d0 to the output; keys in it to the leader's candidate list,
    // both in position order (CTA rank order is position order).  The candidates go out as
    // asynchronous stores counted on the leader's barrier: no cluster barrier waits for
    // them, nor for the output writes ----
    const uint32_t bar = dsmem_addr(&sm.cand_bar, 0);
    const uint32_t lt = (1u << lane) - 1u;
    for (int base = lo; base < hi; base += 32) {
      const int i = base + lane;
      const uint32_t k = i < hi ? keys[i] : 0u;
      const uint32_t dg = k >> 21;
      const bool up = k != 0u && dg > d0, in = k != 0u && dg == d0;
      const uint32_t bg = __ballot_sync(0xffffffffu, up);
      const uint32_t be = __ballot_sync(0xffffffffu, in);
      if (up) {
        const uint32_t slot = og + __popc(bg & lt);
        if (slot < static_cast<uint32_t>(K)) {  // guards the row against an inconsistent count
          out_idx[slot] = c0 + i;
          if (out_scores) out_scores[slot] = key_score(k);
        }
      }
      if (in) {
        const uint32_t slot = oe + __popc(be & lt);
        if (slot < at_total)  // (a slot past the count would never be waited for)
          dsmem_st_async_v2(dsmem_addr(&cand[slot], 0), make_uint2(k, static_cast<uint32_t>(c0 + i)), bar);
      }
      og += __popc(bg);
      oe += __popc(be);
    }
    if (rank == 0) {
      for (int i = tid; i < kHistBins; i += nt) sm.local[i] = 0;  // the leader's scratch, meanwhile
      if (tid == 0) sm.n_few = 0u;
      // every thread waits for the whole list (bounded: a count that never completes flags
      // TIMEOUT and the row is finished with what arrived)
      if (!tc::mbar_try_wait(&sm.cand_bar, cand_parity)) {
        const uint64_t t0 = tc::global_ns();
        for (uint32_t it = 0; !tc::mbar_try_wait(&sm.cand_bar, cand_parity); ++it) {
          if ((it & 255u) == 255u && tc::global_ns() - t0 > wait_ns) {
            flag(status, DSA_STATUS_TIMEOUT);
            break;
          }
        }
      }
      __syncthreads();  // every thread has read the parity before it moves on
      if (tid == 0) sm.cand_uses += 1u;
      leader_finish(sm, cand, at_total, d0, above0, K, out_idx, out_scores);
    }
    return;
  }

  // ---- crowded top bin: second and third digits through the leader ----
  uint32_t prefix = d0 << 21;
  uint32_t need = static_cast<uint32_t>(K) - above0;
#pragma unroll 1
  for (int lvl = 1; lvl < 3; ++lvl) {
    const int sh = lvl == 1 ? 10 : 0;
    const int width = lvl == 2 ? 10 : 11;
    const uint32_t mask = (1u << width) - 1u;
    const int hsh = sh + width;  // bits above this digit must equal prefix's
    uint32_t* cl_hist = sm.hist[lvl & 1];
    for (int i = tid; i < kHistBins; i += nt) sm.local[i] = 0;
    __syncthreads();
    for (int i = tid; i < len; i += nt) {
      const uint32_t k = keys[i];
      if (k != 0u && (k >> hsh) == (prefix >> hsh)) atomicAdd(&sm.local[(k >> sh) & mask], 1u);
    }
    __syncthreads();
    for (int i = tid; i < kHistBins; i += nt) {
      const uint32_t c = sm.local[i];
      if (c) dsmem_add_u32(dsmem_addr(&cl_hist[i], 0), c);
    }
    cluster_sync();
    if (rank == 0) leader_pick(sm, cl_hist, need, nrank);
    cluster_sync();
    prefix |= sm.bcast[0] << sh;
    need -= sm.bcast[1];
  }
  const uint32_t T = prefix;
  cluster_write_selected(sm, keys, c0, len, T, need, K, out_idx, out_scores, row & 1);  // need >= 1 ties
}

}  // namespace dsa
