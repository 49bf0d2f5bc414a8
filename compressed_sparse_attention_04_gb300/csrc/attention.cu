// Stage 4: shared-K=V sparse attention over the selected entries plus the window.
//
// [P1] "DeepSeek-V4.1 模型结构（2）：序列维度（中），CSA2 的三种模式" (blog.javazero.top),
//      §一层全局注意力算四样东西 item 4: the layer's own query reads the k selected
//      main-KV entries plus the 128 rows of its own sliding window.
// [P2] "DeepSeek v4.1 Flash技术剖析——架构篇" (myhz0606.com), §CSA2-FULL: key and value
//      are one shared vector; the attended set concatenates window rows and top-k entries.
// [P3] "DeepSeek-V4.1-Flash：把百万 Token 的记忆，压缩成一套分级缓存" (junki.cn), §四:
//      p_j = softmax_j(c_j . q / sqrt d), o = sum_j p_j c_j.
//
// attn_flash_kernel (64 heads): a cluster of 1-4 CTAs per query row shares the row's
// attended list (each CTA an equal part of the window rows and of the top-k slots); each CTA
// streams its rows in chunks of 48 through a three-slot ring (16-byte asynchronous gathers
// into a K-major 128-byte-swizzled tile), tcgen05
// computes S = Q C^T (64 heads x 48 rows, K = 512) so that one thread owns one head's
// scores, an online softmax writes P (bf16, a head per row), and tcgen05 accumulates O^T = C^T P^T
// (512 dims x 64 heads) in TMEM, reading the SAME shared tile as the MN-major operand
// (K = V).  The CTAs of a cluster combine their (max, sum, O) through distributed shared
// memory; nothing intermediate goes to global memory.
// Its second instantiation serves stored formats ([P3] §六, §七): FP4 entries (E2M1 with one
// E4M3 scale per 16 channels) and / or FP8 window rows (E4M3 with one power-of-two scale per
// 64 channels) are loaded into registers as 16-byte pieces before the ring slot is free and
// dequantised exactly into the same bf16 tile.
//
// attn_simt_kernel (any H): one CTA per (query row, group of 8 heads), one warp per head.
// Rows of A (top-k slots then window rows) stream through shared memory in tiles of
// 32; lane j scores row j of the tile; an online softmax keeps (max, sum) per head
// and every lane accumulates 16 of the 512 output dims.
#include <algorithm>
#include <atomic>
#include <cooperative_groups.h>

#include "common.cuh"
#include "umma.cuh"

CSA2_DEFINE_ERR_WORD(d_err_attn)

namespace csa2 {
namespace {

constexpr int AT_HG = 8;               // heads per CTA (one warp each)
constexpr int AT_T = AT_HG * 32;
constexpr int AT_TILE = 32;            // rows per tile
constexpr int AT_LD = 512 + 8;         // padded row stride in bf16 elements (1040 B)

struct AttnArgs {
  const uint16_t* q;        // [rows, H, 512]
  int rows, Tq, H, q_pos0, n_hg;
  const uint16_t* kv;       // [B, n_cap, 512]
  int n_cap, n_entries;
  const int32_t* topk;      // [rows, k]
  int k;
  const uint16_t* swa;      // [B, S, 512]
  int S, swa_pos0, window;
  const float* sink;
  float scale;
  uint16_t* out;            // [rows, H, 512]
  float* lse;               // [rows, H]
  const uint8_t* kv_codes;  // FP4 main KV [B, n_cap, 256] (NULL: kv holds bf16 entries)
  const uint8_t* kv_scales; // [B, n_cap, 32]
  const uint8_t* swa_codes; // FP8 window KV [B, S, 512] (NULL: swa holds bf16 rows)
  const uint8_t* swa_scales;// [B, S, 8]
};

__global__ void __launch_bounds__(AT_T) attn_simt_kernel(AttnArgs a) {
  pdl_wait();
  __shared__ __align__(16) uint16_t qs[AT_HG][512];
  __shared__ __align__(16) uint16_t tile[AT_TILE][AT_LD];
  __shared__ int valid[AT_TILE];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x / a.n_hg, hg = blockIdx.x % a.n_hg;
  const int b = row / a.Tq, i = row % a.Tq;
  const long long t = (long long)a.q_pos0 + i;
  const int h = hg * AT_HG + warp;
  const bool head_ok = h < a.H;

  for (int idx = tid; idx < AT_HG * 512; idx += AT_T) {
    const int hh = hg * AT_HG + idx / 512;
    qs[idx / 512][idx % 512] = hh < a.H ? a.q[(size_t(row) * a.H + hh) * 512 + idx % 512] : 0;
  }
  const long long lo = t - a.window + 1 > 0 ? t - a.window + 1 : 0;
  const int n_win = int(t - lo + 1);
  const int n_rows = a.k + n_win;

  float m_run = -INFINITY, l_run = 0.f;
  float o[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) o[u] = 0.f;

  for (int r0 = 0; r0 < n_rows; r0 += AT_TILE) {
    __syncthreads();   // previous tile consumed (and qs ready on the first pass)
    if (tid < AT_TILE) {
      const int j = r0 + tid;
      int ok = 0;
      if (j < a.k) {
        const int e = a.topk[size_t(row) * a.k + j];
        if (e >= a.n_entries) atomicOr(&d_err_attn, ERR_BOUNDS);
        ok = (e >= 0 && e < a.n_entries);
      } else if (j < n_rows) {
        ok = 1;
      }
      valid[tid] = ok;
    }
    __syncthreads();
    // 32 rows x 64 chunks of 16 bytes
    for (int c = tid; c < AT_TILE * 64; c += AT_T) {
      const int rr = c >> 6, cc = c & 63, j = r0 + rr;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (valid[rr]) {
        const uint16_t* src;
        if (j < a.k) {
          const int e = a.topk[size_t(row) * a.k + j];
          src = a.kv + (size_t(b) * a.n_cap + e) * 512;
        } else {
          const long long p = lo + (j - a.k);
          src = a.swa + (size_t(b) * a.S + size_t(p - a.swa_pos0)) * 512;
        }
        v = *reinterpret_cast<const uint4*>(src + cc * 8);
      }
      *reinterpret_cast<uint4*>(&tile[rr][cc * 8]) = v;
    }
    __syncthreads();
    if (!head_ok) continue;
    // logit of row `lane` for head h
    float dot = 0.f;
    const uint4* qv = reinterpret_cast<const uint4*>(qs[warp]);
#pragma unroll 4
    for (int d8 = 0; d8 < 64; ++d8) {
      const uint4 kv = *reinterpret_cast<const uint4*>(&tile[lane][d8 * 8]);
      const uint4 qq = qv[d8];
      const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
      const uint32_t qw[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        dot = fmaf(__uint_as_float(qw[u] << 16), __uint_as_float(kw[u] << 16), dot);
        dot = fmaf(__uint_as_float(qw[u] & 0xFFFF0000u), __uint_as_float(kw[u] & 0xFFFF0000u), dot);
      }
    }
    const float lg = valid[lane] ? dot * a.scale : -INFINITY;
    float tmax = lg;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    const float m_new = fmaxf(m_run, tmax);
    if (m_new == -INFINITY) continue;   // whole tile masked so far (uniform per warp)
    const float corr = expf(m_run - m_new);
    const float p = expf(lg - m_new);
    float psum = p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
    l_run = l_run * corr + psum;
    m_run = m_new;
#pragma unroll
    for (int u = 0; u < 16; ++u) o[u] *= corr;
    for (int j = 0; j < AT_TILE; ++j) {
      const float pj = __shfl_sync(0xffffffffu, p, j);
      const uint4 c0 = *reinterpret_cast<const uint4*>(&tile[j][lane * 16]);
      const uint4 c1 = *reinterpret_cast<const uint4*>(&tile[j][lane * 16 + 8]);
      const uint32_t wv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        o[2 * u] = fmaf(pj, __uint_as_float(wv[u] << 16), o[2 * u]);
        o[2 * u + 1] = fmaf(pj, __uint_as_float(wv[u] & 0xFFFF0000u), o[2 * u + 1]);
      }
    }
  }
  if (!head_ok) return;
  if (a.sink) {
    const float sk = a.sink[h];
    const float m_f = fmaxf(m_run, sk);
    const float corr = expf(m_run - m_f);
    l_run = l_run * corr + expf(sk - m_f);
#pragma unroll
    for (int u = 0; u < 16; ++u) o[u] *= corr;
    m_run = m_f;
  }
  const float inv = 1.0f / l_run;
  uint32_t packed[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    __nv_bfloat162 v2 = __floats2bfloat162_rn(o[2 * u] * inv, o[2 * u + 1] * inv);
    packed[u] = *reinterpret_cast<uint32_t*>(&v2);
  }
  uint16_t* dst = a.out + (size_t(row) * a.H + h) * 512 + lane * 16;
  *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  *reinterpret_cast<uint4*>(dst + 8) = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  if (a.lse && lane == 0) a.lse[size_t(row) * a.H + h] = m_run + logf(l_run);
}


// ---------------------------------------------------------------- pipelined tensor-core
// attention (64 heads).  The CTAs of one cluster share a row's attended list: CTA r takes
// its part of the window rows followed by its part of the top-k slots (window rows first:
// the first chunk's copies need no top-k index), cut into chunks of 48 rows, and the CTAs
// merge their partial results through distributed shared memory.  Per chunk:
//   S   = Q C^T     (M = 64 heads, N = 48 rows, K = 512)   -> TMEM, one head per lane,
//                    so each head's softmax runs inside one thread;
//   O^T += C^T P^T  (M = 4 x 128 dims, N = 64 heads, K = 48 rows) -> TMEM,
// reading the SAME shared tile of C (K = V) as a K-major and an MN-major operand.
// The running maximum is only moved when a chunk exceeds it by more than 2^8 (probabilities
// then stay below 256, exact in float32 sums); moving it rescales that head's columns of
// O^T in TMEM after the previous chunk's products have landed.
constexpr int AF_CH = 48;                              // rows per chunk
constexpr int AF_SLOTS = 3;                            // KV ring depth (chunks)
constexpr int AF_T = 288;                              // 4 copy + 4 softmax + 1 MMA warp
constexpr uint32_t AF_KV_BYTES = AF_CH * 1024;         // 48 KB per ring slot
constexpr uint32_t AF_ATOM = AF_CH * 128;              // one 64-dim atom column of a slot
constexpr uint32_t AF_Q_BYTES = 64 * 1024;
// P: 64 heads x 48 rows, K-major without swizzle: 8-head x 8-row core matrices of 128 B,
// K (rows) direction 128 B apart, 8-head groups AF_P_SBO apart
constexpr uint32_t AF_P_SBO = (AF_CH / 8) * 128;
constexpr uint32_t AF_P_BYTES = 8 * AF_P_SBO;          // 6 KB per P buffer
constexpr uint32_t AF_SMEM = AF_SLOTS * AF_KV_BYTES + AF_Q_BYTES + 2 * AF_P_BYTES + 1024;
// Quantised rows (FP4 entries, FP8 window rows) are loaded into registers as 16-byte pieces,
// at most AF_PC per copy thread and round (one round per chunk of FP4 entries, two for a
// chunk of FP8 window rows), then dequantised into the tile.
constexpr int AF_PC = 12;
constexpr int AF_HALF = AF_CH / 2;                     // rows per lane (two lanes per head)
// S: 2 buffers x 2 K-halves x 64 columns (the two halves are independent accumulators so
// that consecutive MMAs do not wait on each other); O^T: 4 x 64 columns
constexpr uint32_t AF_S_COL = 0, AF_O_COL = 256;
constexpr float AF_LAZY = 8.f;                         // log2 slack before the max moves
constexpr int AF_MAX_SPLIT = 4;

struct AttnFlashArgs {
  AttnArgs a;
  int n_split;        // CTAs per row (cluster size)
};

// Shared-memory descriptor without swizzle: 8-row x 16-byte core matrices, LBO = stride
// between core matrices along K, SBO = stride between 8-row groups.
__device__ __forceinline__ uint64_t desc_noswz(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  return d;
}
// 2^x by the MUFU approximation (relative error about 2^-22; the probabilities are rounded
// to bf16 for the products, and the sums use the same values).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Read-only global loads kept in program order with the other volatile statements (the
// slot wait), so that they are in flight while the copy thread waits for a free slot.
__device__ __forceinline__ uint4 ld_v4_early(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_u16_early(const uint8_t* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_u8_early(const uint8_t* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
// Named barrier over n threads.
__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}
// Channels 8g .. 8g + 7 of an FP8 window row as bf16: E4M3 code bytes (channel 8g + i in
// byte i) times the group's 2^(scale byte - 127).  Pairs go through the E4M3x2 -> f16x2
// conversion (exact), then float32, then bf16 (exact: 4 significant bits).
__device__ __forceinline__ uint4 fp8_piece_bf16(uint2 codes, uint32_t scale_byte) {
  const float sc = __uint_as_float(scale_byte << 23);
  uint32_t w[4];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const uint16_t pair = uint16_t(((x < 2 ? codes.x : codes.y) >> (16 * (x & 1))) & 0xFFFFu);
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(f.x * sc, f.y * sc);
    w[x] = *reinterpret_cast<const uint32_t*>(&b2);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
// Channels 8g .. 8g + 7 of an FP4 entry as bf16: E2M1 codes (channel 8g + 2i in the low
// nibble of byte i) times the group's E4M3 scale; the f16 product is exact (at most 6
// significant bits, 2^-10 .. 2688), and so is its bf16 value.
__device__ __forceinline__ uint4 fp4_piece_bf16(uint32_t codes, uint32_t scale_byte) {
  uint32_t s2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2) : "h"(uint16_t(scale_byte)));
  const __half sc = __low2half(*reinterpret_cast<const __half2*>(&s2));
  const __half2 sc2 = __halves2half2(sc, sc);
  uint32_t w[4];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(h2) : "r"((codes >> (8 * x)) & 0xFFu));
    const __half2 prod = __hmul2(*reinterpret_cast<const __half2*>(&h2), sc2);
    const float2 f = __half22float2(prod);
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(f.x, f.y);
    w[x] = *reinterpret_cast<const uint32_t*>(&b2);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
// Bring `bytes` (a multiple of 16) at p into L2 without waiting for them.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// Named barrier over n threads that also reduces a predicate (and / or) across them.
__device__ __forceinline__ bool bar_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
               "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
               : "=r"(r) : "r"(uint32_t(v)), "r"(id), "r"(n) : "memory");
  return r != 0;
}
__device__ __forceinline__ bool bar_or(int id, int n, bool v) {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
               "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
               : "=r"(r) : "r"(uint32_t(v)), "r"(id), "r"(n) : "memory");
  return r != 0;
}

// Marks a quantised row among the bf16 row sources.
#define kQuantRow (reinterpret_cast<const uint16_t*>(uintptr_t(16)))

template <bool QNT>   // QNT: FP4 entries and / or FP8 window rows
__global__ void __launch_bounds__(AF_T, 1) attn_flash_kernel(AttnFlashArgs u) {
  constexpr int NS = AF_SLOTS;
  pdl_wait();
  namespace cg = cooperative_groups;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* KV = base;                                   // NS x 48 rows (K-major SW128)
  uint8_t* Qs = base + NS * AF_KV_BYTES;                // 64 heads (K-major SW128)
  uint8_t* Ps = Qs + AF_Q_BYTES;                        // 2 x P (64 heads x 64 rows, K-major)
  // after the last chunk: partial O^T tiles pushed by the cluster's CTAs to the tile's owner,
  // [slot = source rank][owned tile][head][dim] (KV ring and Q, 192 KB)
  float* Obuf = reinterpret_cast<float*>(KV);
  __shared__ const uint16_t* row_src[NS][AF_CH];   // bf16 row sources (NULL: none)
  __shared__ int row_e[2][AF_CH];                  // (QNT) per copy group: quantised rows, -1 none
  __shared__ unsigned long long row_mask[NS];
  __shared__ __align__(8) uint64_t kv_full[NS], kv_empty[NS];
  __shared__ __align__(8) uint64_t s_full[2], s_empty[2], p_full[2], o_ready;
  __shared__ uint32_t tmem_slot;
  __shared__ float fac[64];                              // per-head factor (rescale / final)
  __shared__ __align__(8) float ml_all[AF_MAX_SPLIT][64][2];   // every CTA's (max, sum), log2 units

  const AttnArgs& a = u.a;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = int(cluster.block_rank());
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = blockIdx.x / u.n_split;
  const int b = row / a.Tq, i = row % a.Tq;
  const long long t = (long long)a.q_pos0 + i;
  const long long lo = t - a.window + 1 > 0 ? t - a.window + 1 : 0;
  // this CTA's rows: window rows w0 .. w1 - 1, then top-k slots k0 .. k1 - 1 (the window
  // first, so that the first chunk's copies need no top-k index)
  const int n_win = int(t - lo + 1);
  const int w0 = int((long long)n_win * rank / u.n_split), nw = int((long long)n_win * (rank + 1) / u.n_split) - w0;
  const int k0 = int((long long)a.k * rank / u.n_split), nk_mine = int((long long)a.k * (rank + 1) / u.n_split) - k0;
  const int n_mine = nw + nk_mine;
  const int n_ch = (n_mine + AF_CH - 1) / AF_CH;
  const float scale_log2 = a.scale * 1.4426950408889634f;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      umma::mbar_init(&kv_full[s], 64);   // the 64 threads of the group that fills it
      umma::mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      umma::mbar_init(&s_full[s], 1);
      umma::mbar_init(&s_empty[s], 4);
      umma::mbar_init(&p_full[s], 4);
    }
    umma::mbar_init(&o_ready, 1);
    umma::mbar_fence_init();
  }
  if (warp == 0) umma::tmem_alloc(&tmem_slot, 512);
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;
  float m_fin = -INFINITY, l_fin = 0.f;   // softmax lanes: this CTA's (max, sum) of their head
  // announce that this CTA runs; the matching wait precedes the first remote access
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  if (warp < 4) {
    // ---------------- copy warps, two groups of two warps: group g fills chunks g, g + 2,
    // g + 4, ... (slot c % 3; group 0 also the queries with chunk 0), waits for its own copies
    // and announces the chunk, so one group waiting for a free slot never holds back the
    // other's announcement.  Thread t < 48 of a group holds the selected entry of row t of
    // the group's next chunk, loaded one chunk ahead.
    const int grp = warp >> 1, gt = tid & 63, gw = warp & 1;
    const bool fp4 = QNT && a.kv_codes != nullptr, fp8w = QNT && a.swa_codes != nullptr;
    auto topk_at = [&](int c) -> int {
      const int j = c * AF_CH + gt;
      return (gt < AF_CH && c < n_ch && j >= nw && j < n_mine) ? a.topk[size_t(row) * a.k + k0 + (j - nw)] : -1;
    };
    int e_next = topk_at(grp);
    for (int c = grp; c < n_ch && ok; c += 2) {
      const int s = c % AF_SLOTS;
      const int e = e_next;
      e_next = topk_at(c + 2);
      // row gt of the chunk: a bf16 source, or the row of a quantised one (qrow), or none
      const int j = c * AF_CH + gt;
      int okr = 0;
      const uint16_t* src = nullptr;
      int qrow = -1;
      if (gt >= AF_CH) {
        // (lanes past the chunk only complete the ballot)
      } else if (j < nw) {
        okr = 1;
        const size_t wr = size_t(b) * a.S + size_t(lo + w0 + j - a.swa_pos0);
        if (fp8w) qrow = int(wr);
        else src = a.swa + wr * 512;
      } else if (j < n_mine) {
        if (e >= a.n_entries) atomicOr(&d_err_attn, ERR_BOUNDS);
        if (e >= 0 && e < a.n_entries) {
          okr = 1;
          if (fp4) qrow = int(size_t(b) * a.n_cap + e);
          else src = a.kv + (size_t(b) * a.n_cap + e) * 512;
        }
      }
      const int r_w = max(0, min(AF_CH, nw - c * AF_CH));   // the chunk's window rows come first
      // (QNT) the chunk's quantised rows as 16-byte pieces, 32 per FP8 window row and 16 per
      // FP4 entry, window rows first; piece idx of the chunk goes to thread idx % 64, at most
      // AF_PC per thread and round, held in registers from before the slot is free
      const int pw = fp8w ? 32 : 0, pm = fp4 ? 16 : 0;
      const int n_pc = r_w * pw + (AF_CH - r_w) * pm;
      uint4 pc[AF_PC];
      uint32_t psc[AF_PC];
      auto piece_at = [&](int idx, int& r, int& p) {
        if (idx < r_w * pw) {
          r = idx >> 5;
          p = idx & 31;
        } else {
          const int i2 = idx - r_w * pw;
          r = r_w + (i2 >> 4);
          p = i2 & 15;
        }
      };
      auto load_round = [&](int base) {   // codes and the scales they need, all in flight
#pragma unroll
        for (int i = 0; i < AF_PC; ++i) {
          const int idx = base + gt + 64 * i;
          if (idx >= n_pc) break;
          int r, p;
          piece_at(idx, r, p);
          const int qr = row_e[grp][r];
          if (qr < 0) continue;
          if (r < r_w) {
            pc[i] = ld_v4_early(a.swa_codes + size_t(qr) * 512 + 16 * p);
            psc[i] = ld_u8_early(a.swa_scales + size_t(qr) * 8 + (p >> 2));
          } else {
            pc[i] = ld_v4_early(a.kv_codes + size_t(qr) * 256 + 16 * p);
            psc[i] = ld_u16_early(a.kv_scales + size_t(qr) * 32 + 2 * p);
          }
        }
      };
      uint8_t* dst = KV + s * AF_KV_BYTES;
      auto store_round = [&](int base) {  // dequantised into the tile (exact in bf16)
#pragma unroll
        for (int i = 0; i < AF_PC; ++i) {
          const int idx = base + gt + 64 * i;
          if (idx >= n_pc) break;
          int r, p;
          piece_at(idx, r, p);
          if (row_e[grp][r] < 0) continue;
          if (r < r_w) {   // channels 16 p .. 16 p + 15, scale group p / 4
            *reinterpret_cast<uint4*>(dst + umma::kmajor_sw128_offset(r, 16 * p, AF_CH)) =
                fp8_piece_bf16(make_uint2(pc[i].x, pc[i].y), psc[i]);
            *reinterpret_cast<uint4*>(dst + umma::kmajor_sw128_offset(r, 16 * p + 8, AF_CH)) =
                fp8_piece_bf16(make_uint2(pc[i].z, pc[i].w), psc[i]);
          } else {         // channels 32 p .. 32 p + 31, scale groups 2 p and 2 p + 1
            const uint32_t s0 = psc[i] & 0xFFu, s1 = (psc[i] >> 8) & 0xFFu;
            *reinterpret_cast<uint4*>(dst + umma::kmajor_sw128_offset(r, 32 * p, AF_CH)) = fp4_piece_bf16(pc[i].x, s0);
            *reinterpret_cast<uint4*>(dst + umma::kmajor_sw128_offset(r, 32 * p + 8, AF_CH)) = fp4_piece_bf16(pc[i].y, s0);
            *reinterpret_cast<uint4*>(dst + umma::kmajor_sw128_offset(r, 32 * p + 16, AF_CH)) = fp4_piece_bf16(pc[i].z, s1);
            *reinterpret_cast<uint4*>(dst + umma::kmajor_sw128_offset(r, 32 * p + 24, AF_CH)) = fp4_piece_bf16(pc[i].w, s1);
          }
        }
      };
      if constexpr (QNT) {
        named_bar(2 + grp, 64);   // the group's previous chunk no longer reads row_e[grp]
        if (gt < AF_CH) row_e[grp][gt] = qrow;
        named_bar(2 + grp, 64);
        load_round(0);
      }
      bool okw = c < AF_SLOTS || umma::mbar_wait(&kv_empty[s], ((c / AF_SLOTS) - 1) & 1, &d_err_attn);
      {   // row sources (both warps of the group, whole warps for the ballot)
        const unsigned m0 = __ballot_sync(0xffffffffu, okr);
        if (okw) {
          if (gt < AF_CH) row_src[s][gt] = qrow >= 0 ? kQuantRow : src;
          if (lane == 0) reinterpret_cast<unsigned*>(&row_mask[s])[gw] = m0;
        }
      }
      // row sources ready; the group agrees on whether the slot wait succeeded
      if (!bar_and(2 + grp, 64, okw)) { ok = false; break; }
      // bf16 rows: 48 rows x 64 pieces of 16 bytes, piece gt of row r; the row sources are
      // read eight at a time before their copies (an asynchronous copy orders the loads after
      // it); a row with no source is zero-filled, a quantised row is written below
#pragma unroll 1
      for (int r0 = 0; r0 < AF_CH; r0 += 8) {
        const uint16_t* sp[8];
#pragma unroll
        for (int u2 = 0; u2 < 8; ++u2) sp[u2] = row_src[s][r0 + u2];
#pragma unroll
        for (int u2 = 0; u2 < 8; ++u2) {
          if (QNT && sp[u2] == kQuantRow) continue;
          umma::cp_async16(dst + umma::kmajor_sw128_offset(r0 + u2, gt * 8, AF_CH),
                           sp[u2] ? sp[u2] + gt * 8 : a.q, sp[u2] ? 16u : 0u);
        }
      }
      if constexpr (QNT) {
        store_round(0);
        for (int base = 64 * AF_PC; base < n_pc; base += 64 * AF_PC) {   // (FP8 window chunks)
          load_round(base);
          store_round(base);
        }
      }
      {   // while this chunk is in flight: the rows of the group's next chunk into L2
        const int jn = (c + 2) * AF_CH + gt;
        if (gt < AF_CH && c + 2 < n_ch && jn < n_mine) {
          if (jn < nw) {
            const size_t wr = size_t(b) * a.S + size_t(lo + w0 + jn - a.swa_pos0);
            if (fp8w) prefetch_l2(a.swa_codes + wr * 512, 512);   // (8 scale bytes: too short)
            else prefetch_l2(a.swa + wr * 512, 1024);
          } else if (e_next >= 0 && e_next < a.n_entries) {
            const size_t er = size_t(b) * a.n_cap + e_next;
            if (fp4) {
              prefetch_l2(a.kv_codes + er * 256, 256);
              prefetch_l2(a.kv_scales + er * 32, 32);
            } else {
              prefetch_l2(a.kv + er * 512, 1024);
            }
          }
        }
      }
      if (c <= 1) {
        // the queries come with the first chunk of each group: heads 0..31 with chunk 0,
        // heads 32..63 with chunk 1 (all 64 with chunk 0 when there is no chunk 1)
        const uint16_t* qrow_p = a.q + size_t(row) * 64 * 512;
        const int h0 = c == 0 ? 0 : 32, nh = (c == 0 && n_ch > 1) ? 32 : 64 - h0;
#pragma unroll 4
        for (int rep = 0; rep < nh; ++rep) {
          const int uidx = rep * 64 + gt, h = h0 + (uidx >> 6), ch = uidx & 63;
          umma::cp_async16(Qs + umma::kmajor_sw128_offset(h, ch * 8, 64), qrow_p + h * 512 + ch * 8, 16u);
        }
      }
      umma::cp_async_commit();
      umma::cp_async_wait_all();        // this thread's copies of chunk c landed
      umma::fence_proxy_async();
      umma::mbar_arrive(&kv_full[s]);
    }
  } else if (warp < 8) {
    // ---------------- softmax warps: warp q holds heads 16 q .. 16 q + 15 in TMEM lanes
    // 0..15; lane l < 16 then takes rows 0..23 of head 16 q + l and lane l + 16 rows 24..47
    // (handed over by shuffles), so the whole warp shares the work.
    const int q = warp & 3, h = 16 * q + (lane & 15);
    const bool head_lane = lane < 16;
    const int half = lane >> 4;
    const uint32_t lane_addr = uint32_t(32 * q) << 16;
    float m_used = -INFINITY, l = 0.f;
    for (int c = 0; c < n_ch && ok; ++c) {
      const int s = c & 1;
      bool okc = __all_sync(0xffffffffu, umma::mbar_wait(&s_full[s], (c >> 1) & 1, &d_err_attn));
      if (!bar_and(1, 128, okc)) { ok = false; break; }
      umma::fence_after();
      float sv[AF_HALF];   // this lane's 24 rows of its head (log2 units, masked)
      {
        uint32_t v0[32], v1[32], w0[32], w1[32];   // K halves, columns 0..31 | 32..63
        umma::tmem_ld32(tmem + lane_addr + AF_S_COL + 128 * s, v0);
        umma::tmem_ld32(tmem + lane_addr + AF_S_COL + 128 * s + 32, v1);
        umma::tmem_ld32(tmem + lane_addr + AF_S_COL + 128 * s + 64, w0);
        umma::tmem_ld32(tmem + lane_addr + AF_S_COL + 128 * s + 96, w1);
        umma::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < AF_HALF; ++j) {
          const float lo_rows = __uint_as_float(v0[j]) + __uint_as_float(w0[j]);
          const int jh = AF_HALF + j;   // row of the upper half (24..47)
          const float hi_rows = jh < 32 ? __uint_as_float(v0[jh < 32 ? jh : 0]) + __uint_as_float(w0[jh < 32 ? jh : 0])
                                        : __uint_as_float(v1[jh >= 32 ? jh - 32 : 0]) +
                                              __uint_as_float(w1[jh >= 32 ? jh - 32 : 0]);
          const float moved = __shfl_sync(0xffffffffu, hi_rows, lane & 15);
          sv[j] = half ? moved : lo_rows;
        }
      }
      umma::fence_before();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&s_empty[s]);
      constexpr unsigned half_bits = (1u << AF_HALF) - 1u;
      const unsigned mask = unsigned(row_mask[c % NS] >> (half * AF_HALF)) & half_bits;
      float cmx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) cmx[u] = -INFINITY;
      if (mask == half_bits) {
#pragma unroll
        for (int j = 0; j < AF_HALF; ++j) {
          sv[j] *= scale_log2;
          cmx[j & 7] = fmaxf(cmx[j & 7], sv[j]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < AF_HALF; ++j) {
          sv[j] = ((mask >> j) & 1u) ? sv[j] * scale_log2 : -INFINITY;
          cmx[j & 7] = fmaxf(cmx[j & 7], sv[j]);
        }
      }
      float cm = fmaxf(fmaxf(fmaxf(cmx[0], cmx[1]), fmaxf(cmx[2], cmx[3])),
                       fmaxf(fmaxf(cmx[4], cmx[5]), fmaxf(cmx[6], cmx[7])));
      cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));   // the head's maximum
      // move the running max only when this chunk exceeds it by more than AF_LAZY
      float f = 1.f;
      if (cm > m_used + AF_LAZY || (m_used == -INFINITY && cm != -INFINITY)) {
        f = m_used == -INFINITY ? 0.f : exp2f(m_used - cm);
        m_used = cm;
        l *= f;
      }
      float psx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) psx[u] = 0.f;
      float p[AF_HALF];
      const float msub = m_used == -INFINITY ? INFINITY : m_used;   // all p = 0 before a valid row
#pragma unroll
      for (int j = 0; j < AF_HALF; ++j) {
        p[j] = fast_exp2(sv[j] - msub);
        psx[j & 7] += p[j];
      }
      l += ((psx[0] + psx[1]) + (psx[2] + psx[3])) + ((psx[4] + psx[5]) + (psx[6] + psx[7]));
      // P buffer s is free once the products of chunk c - 2 have completed
      bool okp = c < 2 ||
                 umma::mbar_wait(&kv_empty[(c - 2) % NS], ((c - 2) / NS) & 1, &d_err_attn);
      if (!bar_and(1, 128, okp)) { ok = false; break; }
      // P as the K-major B operand of O^T += C^T P^T (no swizzle): head h's 8-row runs are
      // 16-byte core-matrix rows; this lane writes its 24 rows as three of them
      uint8_t* pb = Ps + s * AF_P_BYTES + (h >> 3) * AF_P_SBO + (h & 7) * 16;
#pragma unroll
      for (int c3 = 0; c3 < AF_HALF / 8; ++c3) {
        uint32_t w[4];
#pragma unroll
        for (int u2 = 0; u2 < 4; ++u2) {
          __nv_bfloat162 v2 = __floats2bfloat162_rn(p[8 * c3 + 2 * u2], p[8 * c3 + 2 * u2 + 1]);
          w[u2] = *reinterpret_cast<uint32_t*>(&v2);
        }
        const int kc = half * (AF_HALF / 8) + c3;   // 8-row group of the chunk
        *reinterpret_cast<uint4*>(pb + kc * 128) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      // heads whose max moved after products were accumulated: rescale their O^T columns
      const bool need = head_lane && f != 1.f && c > 0;
      if (head_lane) fac[h] = need ? f : 1.f;
      if (bar_or(1, 128, need)) {
        // the previous chunk's products must have landed in O^T first
        const bool okr = __all_sync(0xffffffffu,
                                    umma::mbar_wait(&kv_empty[(c - 1) % NS], ((c - 1) / NS) & 1,
                                                    &d_err_attn));
        if (!bar_and(1, 128, okr)) { ok = false; break; }
        umma::fence_after();
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          float fr[32];
#pragma unroll
          for (int x = 0; x < 32; ++x) fr[x] = fac[32 * hf + x];
#pragma unroll 1
          for (int dt = 0; dt < 4; ++dt) {
            uint32_t o[32];
            const uint32_t addr = tmem + lane_addr + AF_O_COL + 64 * dt + 32 * hf;
            umma::tmem_ld32(addr, o);
            umma::tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * fr[x]);
            umma::tmem_st32(addr, o);
          }
        }
        umma::tmem_st_wait();
      }
      umma::fence_proxy_async();
      umma::fence_before();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&p_full[s]);
    }
    m_fin = m_used;
    l_fin = l + __shfl_xor_sync(0xffffffffu, l, 16);   // both halves of the head's rows
  } else if (warp == 8 && lane == 0) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc_s = umma::idesc_f16(64, AF_CH, 1, 0, 0);
    constexpr uint32_t idesc_o = umma::idesc_f16(128, 64, 1, 1, 0);   // A = C^T (MN-major), B = P (K-major)
    const uint32_t kv0 = umma::smem_u32(KV), q0 = umma::smem_u32(Qs), p0 = umma::smem_u32(Ps);
    auto issue_s = [&](int c) {
      const int s = c & 1, ks_ = c % NS;
      if (!umma::mbar_wait(&kv_full[ks_], (c / NS) & 1, &d_err_attn)) return false;
      // the first S also needs the queries' second half, which comes with chunk 1
      if (c == 0 && n_ch > 1 && !umma::mbar_wait(&kv_full[1], 0, &d_err_attn)) return false;
      if (c >= 2 && !umma::mbar_wait(&s_empty[s], ((c >> 1) - 1) & 1, &d_err_attn)) return false;
      umma::fence_after();
      // K steps alternate between the two half accumulators (dims 0-255, 256-511)
      const uint64_t da0 = umma::desc_sw128(q0, 16, 1024);
      const uint64_t db0 = umma::desc_sw128(kv0 + ks_ * AF_KV_BYTES, 16, 1024);
#pragma unroll
      for (int st = 0; st < 16; ++st)
#pragma unroll
        for (int hk = 0; hk < 2; ++hk) {
          const int ks = hk * 16 + st;
          const uint32_t offa = uint32_t(((ks >> 2) * 8192 + (ks & 3) * 32) >> 4);
          const uint32_t offb = uint32_t(((ks >> 2) * AF_ATOM + (ks & 3) * 32) >> 4);
          umma::mma_f16(tmem + AF_S_COL + 128 * s + 64 * hk, da0 + offa, db0 + offb, idesc_s, st > 0);
        }
      umma::commit(&s_full[s]);
      return true;
    };
    // issue whichever is ready: the next chunk's S (its rows landed, its TMEM buffer read
    // out) or the oldest pending P V (its probabilities written)
    int next_s = 0, next_pv = 0;
    uint32_t idle = 0;
    while (next_pv < n_ch) {
      if (next_s < n_ch && next_s <= next_pv + 1) {
        const int c = next_s, s = c & 1;
        if (umma::mbar_test(&kv_full[c % NS], (c / NS) & 1) &&
            (c != 0 || n_ch == 1 || umma::mbar_test(&kv_full[1], 0)) &&
            (c < 2 || umma::mbar_test(&s_empty[s], ((c >> 1) - 1) & 1))) {
          issue_s(c);
          ++next_s;
          idle = 0;
          continue;
        }
      }
      const int c = next_pv, s = c & 1;
      if (next_pv >= next_s || !umma::mbar_test(&p_full[s], (c >> 1) & 1)) {
        if (++idle > (1u << 26)) { atomicOr(&d_err_attn, ERR_TIMEOUT); break; }
        continue;
      }
      idle = 0;
      ++next_pv;
      umma::fence_after();
      // the four dims tiles are independent accumulators: interleave them
      const int ks_ = c % NS;
      const uint64_t pa0 = umma::desc_sw128(kv0 + ks_ * AF_KV_BYTES, AF_ATOM, 1024);
      const uint64_t pb0 = desc_noswz(p0 + s * AF_P_BYTES, 128, AF_P_SBO);
#pragma unroll
      for (int kk = 0; kk < AF_CH / 16; ++kk)
#pragma unroll
        for (int dt = 0; dt < 4; ++dt)
          umma::mma_f16(tmem + AF_O_COL + 64 * dt, pa0 + uint32_t(((2 * dt) * AF_ATOM + kk * 2048) >> 4),
                        pb0 + uint32_t((kk * 256) >> 4), idesc_o, (c > 0 || kk > 0) ? 1u : 0u);
      umma::commit(&kv_empty[ks_]);
    }
    umma::commit(&o_ready);
  }

  // ---------------- merge.  Every CTA pushes its (max, sum) per head to all CTAs of the
  // row and its scaled O^T tiles to each tile's owner (CTA dt % n_split); remote stores
  // only, so no CTA waits on a remote load.  The owner then sums the slots it received.
  __syncthreads();
  if (n_ch > 0 && warp >= 4 && warp < 8) {
    ok = ok && umma::mbar_wait(&o_ready, 0, &d_err_attn);
    umma::fence_after();
  }
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // every peer has started
  if (warp >= 4 && warp < 8 && lane < 16) {
    const int h = 16 * (warp & 3) + lane;
    const float2 mine = make_float2(m_fin, l_fin);
    for (int r = 0; r < u.n_split; ++r)
      *reinterpret_cast<float2*>(cluster.map_shared_rank(&ml_all[rank][h][0], r)) = mine;
  }
  cluster.sync();
  if (tid < 64) {
    const int h = tid;
    const float sk = a.sink ? a.sink[h] * 1.4426950408889634f : -INFINITY;
    float M = sk;
    for (int r = 0; r < u.n_split; ++r) M = fmaxf(M, ml_all[r][h][0]);
    float L = a.sink ? exp2f(sk - M) : 0.f;
    for (int r = 0; r < u.n_split; ++r)
      if (ml_all[r][h][1] > 0.f) L += ml_all[r][h][1] * exp2f(ml_all[r][h][0] - M);
    fac[h] = ml_all[rank][h][1] > 0.f ? exp2f(ml_all[rank][h][0] - M) / L : 0.f;
    if (rank == 0 && a.lse) a.lse[size_t(row) * 64 + h] = (M + log2f(L)) * 0.6931471805599453f;
  }
  __syncthreads();
  const int n_lt = (4 + u.n_split - 1) / u.n_split;   // tile slots per source rank
  // softmax warps: lane = dim 32 q + lane of each 128-dim tile; the factors go to registers
  // first (the compiler cannot tell the stores below from fac[] and would reload it)
  const bool o_warp = warp >= 4 && warp < 8;
  const int q = warp & 3;
  const uint32_t lane_addr = uint32_t(32 * q) << 16;
  float fr[64];
  if (o_warp) {
#pragma unroll
    for (int x = 0; x < 64; ++x) fr[x] = n_ch > 0 ? fac[x] : 0.f;
    // tiles owned by another CTA: scaled O^T to the owner's slot for this rank
    for (int dt = 0; dt < 4; ++dt) {
      if (dt % u.n_split == rank) continue;
      float* dst = cluster.map_shared_rank(Obuf, dt % u.n_split) +
                   size_t((rank * n_lt + dt / u.n_split) * 64) * 128 + 32 * q + lane;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t o[32];
        if (n_ch > 0) {
          umma::tmem_ld32(tmem + lane_addr + AF_O_COL + 64 * dt + 32 * hf, o);
          umma::tmem_ld_wait();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = 0u;
        }
#pragma unroll
        for (int x = 0; x < 32; ++x) dst[(32 * hf + x) * 128] = __uint_as_float(o[x]) * fr[32 * hf + x];
      }
    }
  }
  umma::fence_before();
  cluster.sync();
  // owned tiles: own O^T (TMEM) plus the other CTAs' slots (local shared memory), bf16 out
  if (o_warp) {
    for (int lt = 0; rank + lt * u.n_split < 4; ++lt) {
      const int dt = rank + lt * u.n_split;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.out) + size_t(row) * 64 * 512 +
                            dt * 128 + 32 * q + lane;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t o[32];
        if (n_ch > 0) {
          umma::tmem_ld32(tmem + lane_addr + AF_O_COL + 64 * dt + 32 * hf, o);
          umma::tmem_ld_wait();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = 0u;
        }
        float acc[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) acc[x] = __uint_as_float(o[x]) * fr[32 * hf + x];
        for (int r = 0; r < u.n_split; ++r) {
          if (r == rank) continue;
          const float* src = Obuf + size_t((r * n_lt + lt) * 64 + 32 * hf) * 128 + 32 * q + lane;
          float v[32];
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] = src[x * 128];
#pragma unroll
          for (int x = 0; x < 32; ++x) acc[x] += v[x];
        }
#pragma unroll
        for (int x = 0; x < 32; ++x) orow[(32 * hf + x) * 512] = __float2bfloat16_rn(acc[x]);
      }
    }
  }
  umma::fence_after();
  if (warp == 0) umma::tmem_free(tmem, 512);
}

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" {

size_t csa2_sparse_attn_workspace_size(int B, int Tq, int H, int k, int window) {
  (void)B; (void)Tq; (void)H; (void)k; (void)window;
  return 0;   // partial results are merged on chip
}

}  // extern "C"

namespace {

// All attention entry points: main-KV entries in bf16 (kv_cache) or FP4 (kv_codes /
// kv_scales), window rows in bf16 (swa_kv) or FP8 (swa_codes / swa_scales); the quantised
// formats run on the 64-head tensor-core kernel only.
int sparse_attn_impl(const void* q, int B, int Tq, int H, int q_pos0, const void* kv_cache,
                     const uint8_t* kv_codes, const uint8_t* kv_scales, int n_cap, int n_entries,
                     const int32_t* topk, int k, const void* swa_kv, const uint8_t* swa_codes,
                     const uint8_t* swa_scales, int S, int swa_pos0, int window,
                     const float* sink, float scale, void* out, float* lse_out, void* workspace,
                     size_t ws_bytes, void* stream) {
  const bool fp4 = kv_codes != nullptr || kv_scales != nullptr;
  const bool fp8w = swa_codes != nullptr || swa_scales != nullptr;
  if (!q || !out) return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: null tensor pointer");
  if (fp8w ? (!swa_codes || !swa_scales || swa_kv) : !swa_kv)
    return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: give the window rows either as bf16 or as FP8 codes + scales");
  if (fp4 && (!kv_codes || !kv_scales || kv_cache))
    return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: give the entries either as bf16 or as FP4 codes + scales");
  if (k < 0 || k > CSA2_MAX_TOPK) return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: k=%d out of [0, 2048]", k);
  if (k > 0 && (!topk || (fp4 ? (!kv_codes || !kv_scales) : !kv_cache)))
    return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: k > 0 needs topk and the cache entries");
  if ((fp4 || fp8w) && H != 64)
    return fail(CSA2_ERR_UNSUPPORTED, "sparse_attn: quantised entries or rows need H = 64 (got %d)", H);
  if ((kv_codes && !aligned16(kv_codes)) || (kv_scales && !aligned16(kv_scales)) ||
      (swa_codes && !aligned16(swa_codes)) || (swa_scales && !aligned16(swa_scales)))
    return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: pointers must be 16-byte aligned");
  if ((fp4 && (long long)B * n_cap > 0x7FFFFFFFll) || (fp8w && (long long)B * S > 0x7FFFFFFFll))
    return fail(CSA2_ERR_UNSUPPORTED, "sparse_attn: quantised cache above 2^31 rows");
  if (B <= 0 || Tq <= 0 || H <= 0 || H > 128 || q_pos0 < 0)
    return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: bad shape B=%d Tq=%d H=%d q_pos0=%d", B, Tq, H, q_pos0);
  if (k > 0 && (n_entries < 0 || n_cap < n_entries || n_cap <= 0))
    return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: bad cache shape n_entries=%d n_cap=%d", n_entries, n_cap);
  if (window < 1 || window > 4096) return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: window=%d out of [1, 4096]", window);
  if (S <= 0 || swa_pos0 < 0) return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: bad window cache S=%d swa_pos0=%d", S, swa_pos0);
  const long long first_lo = (long long)q_pos0 - window + 1 > 0 ? (long long)q_pos0 - window + 1 : 0;
  const long long last_t = (long long)q_pos0 + Tq - 1;
  if (first_lo < swa_pos0 || last_t >= (long long)swa_pos0 + S)
    return fail(CSA2_ERR_INVALID_ARG,
                "sparse_attn: window rows of positions %lld..%lld not inside swa_kv [%d, %lld)",
                first_lo, last_t, swa_pos0, (long long)swa_pos0 + S);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: bad scale");
  if (!aligned16(q) || (kv_cache && !aligned16(kv_cache)) || (topk && !aligned16(topk)) ||
      (swa_kv && !aligned16(swa_kv)) || !aligned16(out) || (sink && !aligned16(sink)) ||
      (lse_out && !aligned16(lse_out)))
    return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: pointers must be 16-byte aligned");
  const long long rows = (long long)B * Tq;
  const int n_hg = ceil_div(H, AT_HG);
  if (rows * n_hg > (1ll << 31) - 1) return fail(CSA2_ERR_UNSUPPORTED, "sparse_attn: too many rows");
  AttnArgs aa{(const uint16_t*)q, int(rows), Tq, H, q_pos0, n_hg, (const uint16_t*)kv_cache,
              n_cap, n_entries, topk, k, (const uint16_t*)swa_kv, S, swa_pos0, window, sink,
              scale, (uint16_t*)out, lse_out, kv_codes, kv_scales, swa_codes, swa_scales};
  cudaStream_t st = (cudaStream_t)stream;
  if (H == 64) {
    // tensor-core path: a cluster of n_split CTAs per row (enough CTAs to cover the SMs),
    // partial results merged through distributed shared memory
    (void)workspace; (void)ws_bytes;
    // per device, once: the kernels' shared-memory attribute and the SM count (cached only
    // after both succeeded; concurrent first calls repeat the same settings)
    static std::atomic<int> sms_cache[64];
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return cuda_fail(e0, "sparse_attn: cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(CSA2_ERR_UNSUPPORTED, "sparse_attn: device id");
    int sms = sms_cache[dev].load(std::memory_order_acquire);
    if (sms == 0) {
      e0 = cudaFuncSetAttribute(attn_flash_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(AF_SMEM));
      if (e0 == cudaSuccess)
        e0 = cudaFuncSetAttribute(attn_flash_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(AF_SMEM));
      if (e0 == cudaSuccess) e0 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e0 != cudaSuccess) return cuda_fail(e0, "sparse_attn: attributes");
      sms_cache[dev].store(sms, std::memory_order_release);
    }
    // CTAs per row: all CTAs in one wave, and the estimated time of a row's chunks (about
    // 1.5 us each, per CTA) plus the cluster merge (about 4 us) the smallest
    const int n_ch_max = ceil_div(k + window, AF_CH);
    const int n_fit = std::max(1, std::min(int(sms / rows), AF_MAX_SPLIT));
    int n_split = 1;
    for (int n = 2; n <= n_fit; ++n) {
      const int t_n = 3 * ceil_div(n_ch_max, n) + 8, t_best = 3 * ceil_div(n_ch_max, n_split) + (n_split > 1 ? 8 : 0);
      if (t_n < t_best) n_split = n;
    }
    if (rows * n_split > (1ll << 31) - 1) return fail(CSA2_ERR_UNSUPPORTED, "sparse_attn: too many rows");
    AttnFlashArgs fa{aa, n_split};
    e0 = (fp4 || fp8w)
             ? launch_k(attn_flash_kernel<true>, dim3(unsigned(rows * n_split), 1, 1), dim3(AF_T, 1, 1),
                        AF_SMEM, st, unsigned(n_split), fa)
             : launch_k(attn_flash_kernel<false>, dim3(unsigned(rows * n_split), 1, 1), dim3(AF_T, 1, 1),
                        AF_SMEM, st, unsigned(n_split), fa);
    if (e0 != cudaSuccess) return cuda_fail(e0, "sparse_attn: launch");
    note_launch();
  } else {
    CSA2_LAUNCH("attn_simt launch", attn_simt_kernel, unsigned(rows * n_hg), AT_T, 0, st, aa);
    note_launch();
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "sparse_attn launch");
  return CSA2_OK;
}

}  // namespace

extern "C" {

int csa2_sparse_attn(const void* q, int B, int Tq, int H, int q_pos0, const void* kv_cache,
                     int n_cap, int n_entries, const int32_t* topk, int k, const void* swa_kv,
                     int S, int swa_pos0, int window, const float* sink, float scale, void* out,
                     float* lse_out, void* workspace, size_t ws_bytes, void* stream) {
  return sparse_attn_impl(q, B, Tq, H, q_pos0, kv_cache, nullptr, nullptr, n_cap, n_entries, topk,
                          k, swa_kv, nullptr, nullptr, S, swa_pos0, window, sink, scale, out,
                          lse_out, workspace, ws_bytes, stream);
}

int csa2_sparse_attn_fp4kv(const void* q, int B, int Tq, int H, int q_pos0,
                           const uint8_t* kv_codes, const uint8_t* kv_scales, int n_cap,
                           int n_entries, const int32_t* topk, int k, const void* swa_kv, int S,
                           int swa_pos0, int window, const float* sink, float scale, void* out,
                           float* lse_out, void* workspace, size_t ws_bytes, void* stream) {
  if (!kv_codes || !kv_scales)
    return fail(CSA2_ERR_INVALID_ARG, "sparse_attn_fp4kv: null FP4 cache pointer");
  return sparse_attn_impl(q, B, Tq, H, q_pos0, nullptr, kv_codes, kv_scales, n_cap, n_entries,
                          topk, k, swa_kv, nullptr, nullptr, S, swa_pos0, window, sink, scale, out,
                          lse_out, workspace, ws_bytes, stream);
}

int csa2_sparse_attn_ex(const void* q, int B, int Tq, int H, int q_pos0, const void* kv_cache,
                        const uint8_t* kv_codes, const uint8_t* kv_scales, int n_cap,
                        int n_entries, const int32_t* topk, int k, const void* swa_kv,
                        const uint8_t* swa_codes, const uint8_t* swa_scales, int S, int swa_pos0,
                        int window, const float* sink, float scale, void* out, float* lse_out,
                        void* workspace, size_t ws_bytes, void* stream) {
  return sparse_attn_impl(q, B, Tq, H, q_pos0, kv_cache, kv_codes, kv_scales, n_cap, n_entries,
                          topk, k, swa_kv, swa_codes, swa_scales, S, swa_pos0, window, sink, scale,
                          out, lse_out, workspace, ws_bytes, stream);
}

}  // extern "C"
