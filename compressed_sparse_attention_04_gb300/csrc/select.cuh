// Block-wide exact top-k selection by radix select on order-preserving float keys.
//
// Order: larger key first; among equal keys the lower position first.  Key 0 marks
// an element that does not compete.  The selected positions are emitted in
// ascending position order (a stable scan), then padded with -1 up to k.
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

struct SelectSmem {
  unsigned hist[256];
  int scan[32];
  unsigned prefix, mask;
  int k_rem, n_valid;
};

// key_of(i) -> uint32 key (0 = not competing); emit(pos, i) writes output slot pos.
// Returns the number of selected elements (min(k, #competing)); only valid on all
// threads after the call.
template <int NT, class KeyFn, class EmitFn>
__device__ int radix_topk(int n, int k, KeyFn key_of, EmitFn emit, SelectSmem& sm) {
  const int tid = threadIdx.x;
  int cnt = 0;
  for (int i = tid; i < n; i += NT) cnt += key_of(i) != 0u;
  int tot;
  block_excl_scan<NT>(cnt, sm.scan, tot);
  const int n_valid = tot;
  unsigned kth = 1u;   // threshold key: select key > kth, plus k_rem keys == kth
  int k_rem = 0;
  if (n_valid > k) {
    if (tid == 0) { sm.prefix = 0u; sm.mask = 0u; sm.k_rem = k; }
    __syncthreads();
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int d = tid; d < 256; d += NT) sm.hist[d] = 0u;
      __syncthreads();
      const unsigned prefix = sm.prefix, mask = sm.mask;
      for (int i = tid; i < n; i += NT) {
        const unsigned key = key_of(i);
        if (key != 0u && (key & mask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid == 0) {
        int need = sm.k_rem, cum = 0, d = 255;
        for (; d > 0; --d) {
          if (cum + int(sm.hist[d]) >= need) break;
          cum += int(sm.hist[d]);
        }
        sm.k_rem = need - cum;
        sm.prefix = prefix | (unsigned(d) << shift);
        sm.mask = mask | (255u << shift);
      }
      __syncthreads();
    }
    kth = sm.prefix;
    k_rem = sm.k_rem;
  }
  // emission in position order
  int eq_before = 0, sel_before = 0;
  for (int base = 0; base < n; base += NT) {
    const int i = base + tid;
    unsigned key = (i < n) ? key_of(i) : 0u;
    const bool gt = key != 0u && (n_valid > k ? key > kth : true);
    const bool eq = key != 0u && n_valid > k && key == kth;
    int eq_tot;
    const int eq_rank = eq_before + block_excl_scan<NT>(eq ? 1 : 0, sm.scan, eq_tot);
    const bool sel = gt || (eq && eq_rank < k_rem);
    int sel_tot;
    const int pos = sel_before + block_excl_scan<NT>(sel ? 1 : 0, sm.scan, sel_tot);
    if (sel && pos < k) emit(pos, i);
    eq_before += eq_tot;
    sel_before += sel_tot;
  }
  const int n_sel = n_valid < k ? n_valid : k;
  for (int p = n_sel + tid; p < k; p += NT) emit(p, -1);
  __syncthreads();
  return n_sel;
}

}  // namespace csa2
