// Block-wide exact top-k selection on order-preserving float keys.
//
// Order: larger key first; among equal keys the lower position first.  Key 0 marks
// an element that does not compete.  The selected positions are emitted in
// ascending position order (a stable scan), then padded with -1 up to k.
//
// Radix select with adaptive digits: the competing keys' min and max share their
// high bits, so each pass histograms the (up to) 11 bits just below the prefix that
// all remaining candidates share.  Scores of one row occupy a narrow float range, so
// fixed 8-bit digits from the top would put almost every key into one or two bins
// (serialising the shared-memory atomics); adaptive digits spread them over up to 2048
// bins and finish in at most three passes.
#pragma once

#include "common.cuh"

namespace csa2 {

// Exclusive prefix sum of `v` over the block (NT threads, NT % 32 == 0); returns the
// prefix and writes the block total to `total`.  `scratch` holds NT/32 ints.
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, int* scratch, int& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[wid] = x;
  __syncthreads();
  int wpre = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    const int s = scratch[w];
    if (w < wid) wpre += s;
    tot += s;
  }
  __syncthreads();
  total = tot;
  return wpre + x - v;
}

constexpr int SEL_BINS = 2048;

struct SelectSmem {
  unsigned hist[SEL_BINS];
  int scan[32];
  unsigned red_min[32], red_max[32];
  unsigned prefix;     // high bits shared by the remaining candidates
  int lo_bits;         // number of undetermined low bits
  int k_rem;           // how many more to take from the remaining candidates
  int found;           // bin index found by the scan (-1 = none yet)
};

// The selection threshold: returns kth and sets n_valid (competing keys) and k_rem so that
// the top-k are the keys > kth plus the first k_rem keys == kth.  When n_valid <= k every
// competing key is taken (kth = 1, k_rem = 0).  kth is then the k-th largest key.
template <int NT, class KeyFn>
__device__ unsigned radix_kth(int n, int k, KeyFn key_of, SelectSmem& sm, int& n_valid, int& k_rem) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // count competitors and their key range
  int cnt = 0;
  unsigned kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int i = tid; i < n; i += NT) {
    const unsigned key = key_of(i);
    if (key != 0u) {
      ++cnt;
      kmin = min(kmin, key);
      kmax = max(kmax, key);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) { sm.red_min[wid] = kmin; sm.red_max[wid] = kmax; }
  block_excl_scan<NT>(cnt, sm.scan, n_valid);   // (its barriers also publish red_min/max)
  unsigned kth = 1u;
  k_rem = 0;
  if (n_valid > k) {
    if (tid == 0) {
      unsigned mn = 0xFFFFFFFFu, mx = 0u;
      for (int w = 0; w < NT / 32; ++w) { mn = min(mn, sm.red_min[w]); mx = max(mx, sm.red_max[w]); }
      const unsigned diff = mn ^ mx;
      const int lo = diff ? 32 - __clz(diff) : 0;
      sm.lo_bits = lo;
      sm.prefix = lo >= 32 ? 0u : (mx & ~((1u << lo) - 1u));
      sm.k_rem = k;
    }
    __syncthreads();
    while (true) {
      const int lo = sm.lo_bits;
      if (lo == 0) break;
      const unsigned prefix = sm.prefix;
      const int shift = lo > 11 ? lo - 11 : 0;
      const int nbins = 1 << (lo - shift);
      const unsigned hi_mask = lo >= 32 ? 0u : ~((1u << lo) - 1u);
      for (int d = tid; d < nbins; d += NT) sm.hist[d] = 0u;
      __syncthreads();
      for (int i = tid; i < n; i += NT) {
        const unsigned key = key_of(i);
        if (key != 0u && (key & hi_mask) == prefix)
          atomicAdd(&sm.hist[(key >> shift) & unsigned(nbins - 1)], 1u);
      }
      __syncthreads();
      // find the bin holding the k_rem-th largest remaining key: thread t owns the
      // bins [nbins - (t+1)*per, nbins - t*per) (top-down), one block scan of the
      // per-thread counts locates the owner, which walks its bins
      {
        const int need = sm.k_rem;
        const int per = (nbins + NT - 1) / NT;
        const int hi = nbins - tid * per, lo2 = max(0, hi - per);
        int local = 0;
        for (int d = hi - 1; d >= lo2; --d) local += int(sm.hist[d]);
        int tot_unused;
        const int above = block_excl_scan<NT>(hi > 0 ? local : 0, sm.scan, tot_unused);
        if (hi > 0 && above < need && above + local >= need) {
          int cum = above, d = hi - 1;
          for (; d > lo2; --d) {
            if (cum + int(sm.hist[d]) >= need) break;
            cum += int(sm.hist[d]);
          }
          sm.k_rem = need - cum;
          sm.prefix = prefix | (unsigned(d) << shift);
          sm.lo_bits = shift;
        }
      }
      __syncthreads();
    }
    kth = sm.prefix;
    k_rem = sm.k_rem;
  }
  return kth;
}

// key_of(i) -> uint32 key (0 = not competing); emit(pos, i) writes output slot pos
// (i = -1 for padding).  Returns min(k, #competing).
template <int NT, class KeyFn, class EmitFn>
__device__ int radix_topk(int n, int k, KeyFn key_of, EmitFn emit, SelectSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int n_valid, k_rem;
  const unsigned kth = radix_kth<NT>(n, k, key_of, sm, n_valid, k_rem);
  // emission in position order: warp w owns the contiguous segment [w*seg, (w+1)*seg);
  // pass A counts its '>' and '==' keys, one block scan places the warps, pass B writes.
  constexpr int NW = NT / 32;
  const int seg = ((n + NW - 1) / NW + 31) & ~31;
  const int s0 = wid * seg, s1 = min(n, s0 + seg);
  const bool cut = n_valid > k;
  int gt_w = 0, eq_w = 0;
  for (int base = s0; base < s1; base += 32) {
    const int i = base + lane;
    const unsigned key = i < s1 ? key_of(i) : 0u;
    const bool gt = key != 0u && (cut ? key > kth : true);
    const bool eq = key != 0u && cut && key == kth;
    gt_w += __popc(__ballot_sync(0xffffffffu, gt));
    eq_w += __popc(__ballot_sync(0xffffffffu, eq));
  }
  int eq_tot;
  const int eq_before_w = block_excl_scan<NT>(lane == 0 ? eq_w : 0, sm.scan, eq_tot);
  const int eq_before = __shfl_sync(0xffffffffu, eq_before_w, 0);
  const int take_eq = max(0, min(eq_w, k_rem - eq_before));
  int sel_tot;
  const int sel_before_w = block_excl_scan<NT>(lane == 0 ? gt_w + take_eq : 0, sm.scan, sel_tot);
  int pos_base = __shfl_sync(0xffffffffu, sel_before_w, 0);
  int eq_seen = eq_before;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = s0; base < s1; base += 32) {
    const int i = base + lane;
    const unsigned key = i < s1 ? key_of(i) : 0u;
    const bool gt = key != 0u && (cut ? key > kth : true);
    const bool eq = key != 0u && cut && key == kth;
    const unsigned eq_mask = __ballot_sync(0xffffffffu, eq);
    const bool sel = gt || (eq && eq_seen + __popc(eq_mask & lt_mask) < k_rem);
    const unsigned sel_mask = __ballot_sync(0xffffffffu, sel);
    const int pos = pos_base + __popc(sel_mask & lt_mask);
    if (sel && pos < k) emit(pos, i);
    pos_base += __popc(sel_mask);
    eq_seen += __popc(eq_mask);
  }
  const int n_sel = n_valid < k ? n_valid : k;
  for (int p = n_sel + tid; p < k; p += NT) emit(p, -1);
  __syncthreads();
  return n_sel;
}

}  // namespace csa2

