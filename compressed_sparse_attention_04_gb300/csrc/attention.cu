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
// attn_decode_kernel (H a multiple of 8 up to 64; query rows past H are zero in its 64-row
// query tile): a cluster of 1-4 CTAs per query row shares the row's
// attended list (each CTA an equal part of the window rows and of the top-k slots).  The
// queries and the bf16 window rows arrive by TMA tile loads; the selected entries are
// gathered by 16-byte asynchronous copies into a two-slot ring of 64-row chunks (K-major,
// 128-byte swizzle).  tcgen05 computes S = Q C^T (64 heads x 64 rows, K = 512) so that one
// thread owns one head's scores, an online softmax writes P (bf16, a head per row), and
// tcgen05 accumulates O^T = C^T P^T (512 dims x 64 heads) in TMEM, reading the SAME shared
// tile as the MN-major operand (K = V).  The CTAs of a cluster combine their (max, sum)
// through distributed shared memory and send each other's O^T tiles by bulk copies between
// their shared memories; nothing intermediate goes to global memory.
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
// its part of the window rows, then its part of the top-k slots, in chunks of 64 rows.
// Shared memory holds the 64 queries (64 KB) and two 64-row chunk slots (64 KB each); a
// slot is eight 8 KB planes, plane j holding dims 64 j .. 64 j + 63 of the slot's rows in
// 8-row atoms of 1 KB (K-major, 128-byte swizzle); the queries use the same layout.
// Where the rows come from:
//   queries and bf16 window rows: TMA tile loads (one 64-row x 64-dim box per plane),
//     issued at the start for the first two chunks by the MMA warp;
//   top-k entries (and later window chunks): 16-byte cp.async gathers by two copy groups
//     of 64 threads, group g owning slot g; thread t copies 16-byte piece t of every row;
//   FP4 entries / FP8 window rows: the same groups load the quantised pieces into
//     registers before the slot is free and dequantise them exactly into the tile.
// Per chunk:
//   S   = Q C^T     (M = 64 heads, N = 64 rows, K = 512)   -> TMEM, one head per lane,
//                    so each head's softmax runs inside one thread (two lanes split its rows);
//   O^T += C^T P^T  (M = 4 x 128 dims, N = 64 heads, K = 64 rows) -> TMEM,
// reading the SAME shared tile of C (K = V) as a K-major and an MN-major operand.
// The running maximum is only moved when a chunk exceeds it by more than 2^4 (probabilities
// then stay below 16; a larger slack costs accuracy where one row dominates, since the
// dominant probability is then rounded to bf16 instead of being exactly 1); moving it
// rescales that head's columns of O^T in TMEM after the previous chunk's products have
// landed.  The softmax sum adds the bf16-rounded probabilities the products use.
// Merge: the CTAs exchange their (max, sum) per head through distributed shared memory;
// each scales the O^T tiles that another CTA owns into its own shared memory and sends
// each to its owner with one bulk copy; the owner adds them to its own tiles.
constexpr int AD_CH = 64;                              // rows per chunk
constexpr int AD_SLOTS = 2;                            // chunk slots (one per copy group)
constexpr int AD_T = 288;                              // 4 copy + 4 softmax + 1 MMA warp
constexpr uint32_t AD_PLANE = AD_CH * 128;             // 64 rows x 64 dims: 8 KB
constexpr uint32_t AD_SLOT_BYTES = 8 * AD_PLANE;       // 64 KB per slot
constexpr uint32_t AD_Q_BYTES = 64 * 1024;             // 64 heads, same plane layout
// P: 64 heads x 64 rows, K-major without swizzle: 8-head x 8-row core matrices of 128 B,
// K (rows) direction 128 B apart, 8-head groups AD_P_SBO apart
constexpr uint32_t AD_P_SBO = (AD_CH / 8) * 128;
constexpr uint32_t AD_P_BYTES = 8 * AD_P_SBO;          // 8 KB per P buffer
constexpr uint32_t AD_SMEM = AD_SLOTS * AD_SLOT_BYTES + AD_Q_BYTES + 2 * AD_P_BYTES + 1024;
constexpr uint32_t AD_TILE_BYTES = 64 * 128 * 4;       // one O^T tile: 64 heads x 128 dims f32
// Quantised rows are loaded as 16-byte pieces, AD_PC per copy thread and round: one round
// per chunk of FP4 entries (16 pieces a row), two for a chunk of FP8 window rows (32).
constexpr int AD_PC = 16;
constexpr int AD_HALF = AD_CH / 2;                     // rows per lane (two lanes per head)
constexpr uint32_t AD_S_COL = 0, AD_O_COL = 256;       // S: 2 x 64 columns; O^T: 4 x 64
constexpr float AD_LAZY = 4.f;                         // log2 slack before the max moves
constexpr int AD_MAX_SPLIT = 4;
// named barriers (0 is __syncthreads): copy threads 1, copy groups 2 and 3, softmax 4
constexpr int BAR_COPY = 1, BAR_GROUP = 2, BAR_SOFTMAX = 4;

struct AttnDecodeArgs {
  AttnArgs a;
  int n_split;        // CTAs per row (cluster size)
  int win_tma;        // bf16 window rows through the tensor map
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
// Byte offset of channels ch .. ch + 7 (ch a multiple of 8) of row r inside a slot (or the
// query block): plane ch / 64, 8-row atom r / 8, 16-byte chunk swizzled by r % 8.
__device__ __forceinline__ uint32_t plane_off(int r, int ch) {
  return uint32_t((ch >> 6) * AD_PLANE + (r >> 3) * 1024 + (r & 7) * 128 +
                  ((((ch & 63) >> 3) ^ (r & 7)) << 4));
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

// ---- TMA tile loads, bulk shared-memory copies between the CTAs of a cluster
__device__ __forceinline__ void mbar_expect_tx(void* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
               :: "r"(umma::smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, void* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];"
      :: "r"(umma::smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(umma::smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            void* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];"
      :: "r"(umma::smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(z), "r"(umma::smem_u32(bar))
      : "memory");
}
// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(const void* p, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(umma::smem_u32(p)), "r"(rank));
  return r;
}
// `bytes` from this CTA's shared memory to another CTA's, completing on its mbarrier.
__device__ __forceinline__ void bulk_to_peer(uint32_t dst_cluster, const void* src, uint32_t bytes,
                                             uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(dst_cluster), "r"(umma::smem_u32(src)), "r"(bytes), "r"(bar_cluster) : "memory");
}
// O^T tiles (4 of 128 dims) owned by CTA r of n: dt = r, r + n, ...
__device__ __forceinline__ int tiles_owned(int r, int n) { return (4 - r + n - 1) / n; }

// QNT: FP4 entries and / or FP8 window rows.  H64: exactly 64 heads (the head count is then a
// compile-time constant and nothing is masked); otherwise a.H, a multiple of 8 below 64.
template <bool QNT, bool H64>
__global__ void __launch_bounds__(AD_T, 1) attn_decode_kernel(AttnDecodeArgs u,
                                                              const __grid_constant__ CUtensorMap q_map,
                                                              const __grid_constant__ CUtensorMap swa_map) {
  pdl_wait();
  namespace cg = cooperative_groups;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* KV = base;                                   // 2 slots x 64 rows
  uint8_t* Qs = base + AD_SLOTS * AD_SLOT_BYTES;        // 64 heads
  uint8_t* Ps = Qs + AD_Q_BYTES;                        // 2 x P (64 heads x 64 rows)
  // after the last chunk the slots and the queries (192 KB) hold the merge tiles: first the
  // tiles this CTA sends, then the ones it receives, [source][owned tile][head][dim]
  uint8_t* Mg = base;
  __shared__ int sidx[CSA2_MAX_TOPK];                   // this CTA's top-k slots
  __shared__ const uint16_t* row_src[AD_SLOTS][AD_CH];  // bf16 row sources (NULL: none)
  __shared__ int row_q[AD_SLOTS][AD_CH];                // (QNT) quantised rows, -1 none
  __shared__ unsigned long long row_mask[AD_SLOTS];
  __shared__ __align__(8) uint64_t kv_full[AD_SLOTS], kv_empty[AD_SLOTS];
  __shared__ __align__(8) uint64_t s_full[2], s_empty[2], p_full[2], o_ready, q_full, recv_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ float fac[64];                              // per-head factor (rescale / final)
  // every CTA's (max, sum of the bf16-rounded probabilities, exact sum) per head, log2 units
  __shared__ __align__(16) float ml_all[AD_MAX_SPLIT][64][4];

  const AttnArgs& a = u.a;
  const int NH = H64 ? 64 : a.H;   // heads
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = int(cluster.block_rank());
  const int ns = u.n_split;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = blockIdx.x / ns;
  const int b = row / a.Tq, i = row % a.Tq;
  const long long t = (long long)a.q_pos0 + i;
  const long long lo = t - a.window + 1 > 0 ? t - a.window + 1 : 0;
  // this CTA's rows: window rows w0 .. w0 + nw - 1, then top-k slots k0 .. k0 + nk - 1
  const int n_win = int(t - lo + 1);
  const int w0 = int((long long)n_win * rank / ns), nw = int((long long)n_win * (rank + 1) / ns) - w0;
  const int k0 = int((long long)a.k * rank / ns), nk = int((long long)a.k * (rank + 1) / ns) - k0;
  const int n_wch = (nw + AD_CH - 1) / AD_CH, n_ch = n_wch + (nk + AD_CH - 1) / AD_CH;
  const int n_tma = u.win_tma ? min(n_wch, AD_SLOTS) : 0;   // window chunks loaded by the TMA
  const float scale_log2 = a.scale * 1.4426950408889634f;

  if (tid == 0) {
    for (int s = 0; s < AD_SLOTS; ++s) {
      umma::mbar_init(&kv_full[s], 1);    // the TMA issuer's or a copy group's elected arrive
      umma::mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      umma::mbar_init(&s_full[s], 1);
      umma::mbar_init(&s_empty[s], 4);
      umma::mbar_init(&p_full[s], 4);
    }
    umma::mbar_init(&o_ready, 1);
    umma::mbar_init(&q_full, 1);
    umma::mbar_init(&recv_bar, 1);
    umma::mbar_fence_init();
  }
  if (warp == 0) umma::tmem_alloc(&tmem_slot, 512);
  if (!H64) {   // query rows H..63 of every plane are zero (the TMA fills rows 0..H-1)
    const int zb = (64 - a.H) * 128 / 16;   // 16-byte units per plane (a.H < 64 here)
    for (int u = tid; u < 8 * zb; u += AD_T)
      *reinterpret_cast<uint4*>(Qs + (u / zb) * AD_PLANE + a.H * 128 + (u % zb) * 16) = make_uint4(0, 0, 0, 0);
    umma::fence_proxy_async();
  }
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;
  // softmax lanes: this CTA's (max, rounded sum, exact sum) of their head
  float m_fin = -INFINITY, l_fin = 0.f, e_fin = 0.f;
  // announce that this CTA runs; the matching wait precedes the first remote access
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  if (warp < 4) {
    // ---------------- copy warps.  Group g (warps 2g, 2g + 1) fills the chunks of slot g
    // that the TMA does not: it waits for the slot, gathers the chunk (thread gt copies
    // piece gt of each of its 64 rows), waits for its own copies and announces the chunk.
    for (int j = tid; j < nk; j += 128) sidx[j] = a.topk[size_t(row) * a.k + k0 + j];
    named_bar(BAR_COPY, 128);
    const int grp = warp >> 1, gt = tid & 63, gw = warp & 1;
    const bool fp4 = QNT && a.kv_codes != nullptr, fp8w = QNT && a.swa_codes != nullptr;
    uint8_t* dst = KV + grp * AD_SLOT_BYTES;
    for (int c = grp; c < n_ch && ok; c += AD_SLOTS) {
      if (c < n_tma) continue;
      const int s = grp;
      const bool win = c < n_wch;
      const bool qchunk = QNT && (win ? fp8w : fp4);
      // row gt of the chunk: a bf16 source, a quantised row, or none (zero-filled)
      const int j = win ? c * AD_CH + gt : (c - n_wch) * AD_CH + gt;
      int okr = 0, qrow = -1;
      const uint16_t* src = nullptr;
      if (win) {
        if (j < nw) {
          okr = 1;
          const size_t wr = size_t(b) * a.S + size_t(lo + w0 + j - a.swa_pos0);
          if (fp8w) qrow = int(wr);
          else src = a.swa + wr * 512;
        }
      } else if (j < nk) {
        const int e = sidx[j];
        if (e >= a.n_entries) atomicOr(&d_err_attn, ERR_BOUNDS);
        if (e >= 0 && e < a.n_entries) {
          okr = 1;
          if (fp4) qrow = int(size_t(b) * a.n_cap + e);
          else src = a.kv + (size_t(b) * a.n_cap + e) * 512;
        }
      }
      // (QNT) the chunk's quantised rows as 16-byte pieces: piece idx of the chunk (row
      // idx / ppr) goes to thread idx % 64, AD_PC per thread and round, held in registers
      // from before the slot is free
      const int ppr = win ? 32 : 16;
      uint4 pc[AD_PC];
      uint32_t psc[AD_PC];
      auto load_round = [&](int base_idx) {
#pragma unroll
        for (int x = 0; x < AD_PC; ++x) {
          const int idx = base_idx + gt + 64 * x;
          const int r = idx / ppr, p = idx % ppr;
          const int qr = row_q[s][r];
          if (qr < 0) continue;
          if (win) {
            pc[x] = ld_v4_early(a.swa_codes + size_t(qr) * 512 + 16 * p);
            psc[x] = ld_u8_early(a.swa_scales + size_t(qr) * 8 + (p >> 2));
          } else {
            pc[x] = ld_v4_early(a.kv_codes + size_t(qr) * 256 + 16 * p);
            psc[x] = ld_u16_early(a.kv_scales + size_t(qr) * 32 + 2 * p);
          }
        }
      };
      auto store_round = [&](int base_idx) {   // dequantised into the tile (exact in bf16)
#pragma unroll
        for (int x = 0; x < AD_PC; ++x) {
          const int idx = base_idx + gt + 64 * x;
          const int r = idx / ppr, p = idx % ppr;
          const bool have = row_q[s][r] >= 0;
          if (win) {   // channels 16 p .. 16 p + 15, scale group p / 4
            const uint4 z = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(dst + plane_off(r, 16 * p)) =
                have ? fp8_piece_bf16(make_uint2(pc[x].x, pc[x].y), psc[x]) : z;
            *reinterpret_cast<uint4*>(dst + plane_off(r, 16 * p + 8)) =
                have ? fp8_piece_bf16(make_uint2(pc[x].z, pc[x].w), psc[x]) : z;
          } else {     // channels 32 p .. 32 p + 31, scale groups 2 p and 2 p + 1
            const uint4 z = make_uint4(0, 0, 0, 0);
            const uint32_t s0 = psc[x] & 0xFFu, s1 = (psc[x] >> 8) & 0xFFu;
            *reinterpret_cast<uint4*>(dst + plane_off(r, 32 * p)) = have ? fp4_piece_bf16(pc[x].x, s0) : z;
            *reinterpret_cast<uint4*>(dst + plane_off(r, 32 * p + 8)) = have ? fp4_piece_bf16(pc[x].y, s0) : z;
            *reinterpret_cast<uint4*>(dst + plane_off(r, 32 * p + 16)) = have ? fp4_piece_bf16(pc[x].z, s1) : z;
            *reinterpret_cast<uint4*>(dst + plane_off(r, 32 * p + 24)) = have ? fp4_piece_bf16(pc[x].w, s1) : z;
          }
        }
      };
      if (qchunk) {
        row_q[s][gt] = qrow;
        named_bar(BAR_GROUP + grp, 64);
        load_round(0);
      }
      const bool okw = c < AD_SLOTS || umma::mbar_wait(&kv_empty[s], ((c / AD_SLOTS) - 1) & 1, &d_err_attn);
      {   // row sources and the chunk's row mask (whole warps for the ballot)
        const unsigned m0 = __ballot_sync(0xffffffffu, okr);
        if (okw) {
          row_src[s][gt] = src;
          if (lane == 0) reinterpret_cast<unsigned*>(&row_mask[s])[gw] = m0;
        }
      }
      // row sources ready; the group agrees on whether the slot wait succeeded
      if (!bar_and(BAR_GROUP + grp, 64, okw)) { ok = false; break; }
      if (qchunk) {
        store_round(0);
        for (int base_idx = 64 * AD_PC; base_idx < AD_CH * ppr; base_idx += 64 * AD_PC) {   // (FP8)
          load_round(base_idx);
          store_round(base_idx);
        }
      } else {
        // bf16 rows: 64 rows x 64 pieces of 16 bytes, piece gt of row r; the row sources are
        // read eight at a time before their copies; a row with no source is zero-filled
#pragma unroll 1
        for (int r0 = 0; r0 < AD_CH; r0 += 8) {
          const uint16_t* sp[8];
#pragma unroll
          for (int u2 = 0; u2 < 8; ++u2) sp[u2] = row_src[s][r0 + u2];
#pragma unroll
          for (int u2 = 0; u2 < 8; ++u2)
            umma::cp_async16(dst + plane_off(r0 + u2, gt * 8), sp[u2] ? sp[u2] + gt * 8 : a.q,
                             sp[u2] ? 16u : 0u);
        }
        umma::cp_async_commit();
        umma::cp_async_wait_all();        // this thread's copies of chunk c landed
      }
      umma::fence_proxy_async();
      named_bar(BAR_GROUP + grp, 64);     // every thread's part of the chunk is in place
      if (gt == 0) umma::mbar_arrive(&kv_full[s]);
    }
  } else if (warp < 8) {
    // ---------------- softmax warps: warp q holds heads 16 q .. 16 q + 15 in TMEM lanes
    // 0..15; lane l < 16 then takes rows 0..31 of head 16 q + l and lane l + 16 rows 32..63
    // (handed over by shuffles), so the whole warp shares the work.
    const int q = warp & 3, h = 16 * q + (lane & 15);
    const bool head_lane = lane < 16;
    const int half = lane >> 4;
    const uint32_t lane_addr = uint32_t(32 * q) << 16;
    float m_used = -INFINITY, l = 0.f, le = 0.f;   // sums of the rounded / exact probabilities
    for (int c = 0; c < n_ch && ok; ++c) {
      const int s = c & 1;
      const bool okc = __all_sync(0xffffffffu, umma::mbar_wait(&s_full[s], (c >> 1) & 1, &d_err_attn));
      if (!bar_and(BAR_SOFTMAX, 128, okc)) { ok = false; break; }
      umma::fence_after();
      float sv[AD_HALF];   // this lane's 32 rows of its head (log2 units, masked)
      {
        uint32_t v0[32], v1[32];   // rows 0..31 | 32..63 of the lane's head (lanes < 16)
        umma::tmem_ld32(tmem + lane_addr + AD_S_COL + 64 * s, v0);
        umma::tmem_ld32(tmem + lane_addr + AD_S_COL + 64 * s + 32, v1);
        umma::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < AD_HALF; ++j) {
          const float moved = __shfl_sync(0xffffffffu, __uint_as_float(v1[j]), lane & 15);
          sv[j] = half ? moved : __uint_as_float(v0[j]);
        }
      }
      umma::fence_before();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&s_empty[s]);
      const unsigned mask = unsigned(row_mask[s] >> (half * AD_HALF));
      float cmx[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) cmx[x] = -INFINITY;
      if (mask == 0xffffffffu) {
#pragma unroll
        for (int j = 0; j < AD_HALF; ++j) {
          sv[j] *= scale_log2;
          cmx[j & 7] = fmaxf(cmx[j & 7], sv[j]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < AD_HALF; ++j) {
          sv[j] = ((mask >> j) & 1u) ? sv[j] * scale_log2 : -INFINITY;
          cmx[j & 7] = fmaxf(cmx[j & 7], sv[j]);
        }
      }
      float cm = fmaxf(fmaxf(fmaxf(cmx[0], cmx[1]), fmaxf(cmx[2], cmx[3])),
                       fmaxf(fmaxf(cmx[4], cmx[5]), fmaxf(cmx[6], cmx[7])));
      cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));   // the head's maximum
      // move the running max only when this chunk exceeds it by more than AD_LAZY
      float f = 1.f;
      if (cm > m_used + AD_LAZY || (m_used == -INFINITY && cm != -INFINITY)) {
        f = m_used == -INFINITY ? 0.f : exp2f(m_used - cm);
        m_used = cm;
        l *= f;
        le *= f;
      }
      // probabilities rounded to bf16 for the products; the output's normaliser adds the
      // same rounded values (so each output is an exact convex combination of its rows),
      // the log-sum-exp the exact ones
      float psx[4], pex[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) psx[x] = pex[x] = 0.f;
      uint32_t pk[AD_HALF / 2];
      const float msub = m_used == -INFINITY ? INFINITY : m_used;   // all p = 0 before a valid row
#pragma unroll
      for (int j = 0; j < AD_HALF; j += 2) {
        const float p0 = fast_exp2(sv[j] - msub), p1 = fast_exp2(sv[j + 1] - msub);
        const __nv_bfloat162 v2 = __floats2bfloat162_rn(p0, p1);
        pk[j >> 1] = *reinterpret_cast<const uint32_t*>(&v2);
        const float2 r2 = __bfloat1622float2(v2);
        psx[(j >> 1) & 3] += r2.x + r2.y;
        pex[(j >> 1) & 3] += p0 + p1;
      }
      l += (psx[0] + psx[1]) + (psx[2] + psx[3]);
      le += (pex[0] + pex[1]) + (pex[2] + pex[3]);
      // P buffer s is free once the products of chunk c - 2 have completed
      const bool okp = c < 2 || umma::mbar_wait(&kv_empty[s], ((c - 2) >> 1) & 1, &d_err_attn);
      if (!bar_and(BAR_SOFTMAX, 128, okp)) { ok = false; break; }
      // P as the K-major B operand of O^T += C^T P^T (no swizzle): head h's 8-row runs are
      // 16-byte core-matrix rows; this lane writes its 32 rows as four of them
      uint8_t* pb = Ps + s * AD_P_BYTES + (h >> 3) * AD_P_SBO + (h & 7) * 16;
#pragma unroll
      for (int c4 = 0; c4 < AD_HALF / 8; ++c4) {
        const int kc = half * (AD_HALF / 8) + c4;   // 8-row group of the chunk
        *reinterpret_cast<uint4*>(pb + kc * 128) =
            make_uint4(pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
      }
      // heads whose max moved after products were accumulated: rescale their O^T columns
      const bool need = head_lane && f != 1.f && c > 0;
      if (head_lane) fac[h] = need ? f : 1.f;
      if (bar_or(BAR_SOFTMAX, 128, need)) {
        // the previous chunk's products must have landed in O^T first
        const bool okr = __all_sync(0xffffffffu,
                                    umma::mbar_wait(&kv_empty[(c - 1) & 1], ((c - 1) >> 1) & 1,
                                                    &d_err_attn));
        if (!bar_and(BAR_SOFTMAX, 128, okr)) { ok = false; break; }
        umma::fence_after();
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          float fr[32];
#pragma unroll
          for (int x = 0; x < 32; ++x) fr[x] = fac[32 * hf + x];
#pragma unroll 1
          for (int dt = 0; dt < 4; ++dt) {
            uint32_t o[32];
            const uint32_t addr = tmem + lane_addr + AD_O_COL + 64 * dt + 32 * hf;
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
    e_fin = le + __shfl_xor_sync(0xffffffffu, le, 16);
  } else if (warp == 8 && lane == 0) {
    // ---------------- TMA and MMA issuer.  First the queries and the window chunks the
    // TMA loads (their row masks are written here, before their slot is announced).
    mbar_expect_tx(&q_full, uint32_t(NH) * 1024u);   // H heads x 512 dims x 2 bytes
#pragma unroll 1
    for (int j = 0; j < 8; ++j) tma_load_2d(Qs + j * AD_PLANE, &q_map, 64 * j, row * NH, &q_full);
#pragma unroll 1
    for (int c = 0; c < n_tma; ++c) {
      const int valid = min(AD_CH, nw - AD_CH * c);
      row_mask[c] = valid >= 64 ? ~0ull : ((1ull << valid) - 1ull);
      mbar_expect_tx(&kv_full[c], AD_SLOT_BYTES);
      const int y = int(lo + w0 + AD_CH * c - a.swa_pos0);
#pragma unroll 1
      for (int j = 0; j < 8; ++j)
        tma_load_3d(KV + c * AD_SLOT_BYTES + j * AD_PLANE, &swa_map, 64 * j, y, b, &kv_full[c]);
    }
    constexpr uint32_t idesc_s = umma::idesc_f16(64, AD_CH, 1, 0, 0);
    constexpr uint32_t idesc_o = umma::idesc_f16(128, 64, 1, 1, 0);   // A = C^T (MN-major), B = P (K-major)
    const uint32_t kv0 = umma::smem_u32(KV), q0 = umma::smem_u32(Qs), p0 = umma::smem_u32(Ps);
    auto issue_s = [&](int c) {
      const int s = c & 1;
      umma::fence_after();
      const uint64_t da0 = umma::desc_sw128(q0, 16, 1024);
      const uint64_t db0 = umma::desc_sw128(kv0 + s * AD_SLOT_BYTES, 16, 1024);
#pragma unroll
      for (int ks = 0; ks < 32; ++ks) {
        const uint32_t off = uint32_t(((ks >> 2) * AD_PLANE + (ks & 3) * 32) >> 4);
        umma::mma_f16(tmem + AD_S_COL + 64 * s, da0 + off, db0 + off, idesc_s, ks > 0 ? 1u : 0u);
      }
      umma::commit(&s_full[s]);
    };
    auto issue_pv = [&](int c) {
      const int s = c & 1;
      umma::fence_after();
      // the four dims tiles are independent accumulators: interleave them
      const uint64_t pa0 = umma::desc_sw128(kv0 + s * AD_SLOT_BYTES, AD_PLANE, 1024);
      const uint64_t pb0 = desc_noswz(p0 + s * AD_P_BYTES, 128, AD_P_SBO);
#pragma unroll
      for (int kk = 0; kk < AD_CH / 16; ++kk)
#pragma unroll
        for (int dt = 0; dt < 4; ++dt)
          umma::mma_f16(tmem + AD_O_COL + 64 * dt, pa0 + uint32_t(((2 * dt) * AD_PLANE + kk * 2048) >> 4),
                        pb0 + uint32_t((kk * 256) >> 4), idesc_o, (c > 0 || kk > 0) ? 1u : 0u);
      umma::commit(&kv_empty[s]);   // slot s and P buffer s free again
    };
    // issue whichever is ready: the next chunk's S (its rows landed, its TMEM buffer read
    // out, the queries there) or the oldest pending P V (its probabilities written)
    int next_s = 0, next_pv = 0;
    uint32_t idle = 0;
    while (next_pv < n_ch) {
      if (next_s < n_ch && next_s <= next_pv + 1) {
        const int c = next_s, s = c & 1;
        if (umma::mbar_test(&kv_full[s], (c >> 1) & 1) && (c != 0 || umma::mbar_test(&q_full, 0)) &&
            (c < 2 || umma::mbar_test(&s_empty[s], ((c >> 1) - 1) & 1))) {
          issue_s(c);
          ++next_s;
          idle = 0;
          continue;
        }
      }
      const int c = next_pv;
      if (next_pv < next_s && umma::mbar_test(&p_full[c & 1], (c >> 1) & 1)) {
        issue_pv(c);
        ++next_pv;
        idle = 0;
        continue;
      }
      if (++idle > (1u << 26)) { atomicOr(&d_err_attn, ERR_TIMEOUT); break; }
    }
    umma::commit(&o_ready);
  }

  // ---------------- merge
  __syncthreads();
  const bool o_warp = warp >= 4 && warp < 8;
  if (n_ch > 0 && o_warp) {
    ok = ok && umma::mbar_wait(&o_ready, 0, &d_err_attn);
    umma::fence_after();
  }
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // every peer has started
  const int n_own = tiles_owned(rank, ns), n_out = 4 - n_own;
  if (ns > 1 && tid == 0) mbar_expect_tx(&recv_bar, uint32_t(n_own * (ns - 1)) * AD_TILE_BYTES);
  if (o_warp && lane < 16) {
    const int h = 16 * (warp & 3) + lane;
    const float4 mine = make_float4(m_fin, l_fin, e_fin, 0.f);
    for (int r = 0; r < ns; ++r)
      *reinterpret_cast<float4*>(cluster.map_shared_rank(&ml_all[rank][h][0], r)) = mine;
  }
  cluster.sync();
  if (tid < 64) {
    const int h = tid;
    const float sk = a.sink && h < NH ? a.sink[h] * 1.4426950408889634f : -INFINITY;
    float M = sk;
    for (int r = 0; r < ns; ++r) M = fmaxf(M, ml_all[r][h][0]);
    float L = a.sink ? exp2f(sk - M) : 0.f, Le = L;
    for (int r = 0; r < ns; ++r)
      if (ml_all[r][h][1] > 0.f) {
        const float g = exp2f(ml_all[r][h][0] - M);
        L += ml_all[r][h][1] * g;
        Le += ml_all[r][h][2] * g;
      }
    fac[h] = ml_all[rank][h][1] > 0.f ? exp2f(ml_all[rank][h][0] - M) / L : 0.f;
    if (rank == 0 && a.lse && h < NH) a.lse[size_t(row) * NH + h] = (M + log2f(Le)) * 0.6931471805599453f;
  }
  __syncthreads();
  // softmax warps: lane = dim 32 q + lane of each 128-dim tile; the factors go to registers
  // first (the compiler cannot tell the stores below from fac[] and would reload it)
  const int q = warp & 3;
  const uint32_t lane_addr = uint32_t(32 * q) << 16;
  float fr[64];
  if (o_warp) {
#pragma unroll
    for (int x = 0; x < 64; ++x) fr[x] = n_ch > 0 ? fac[x] : 0.f;
    // tiles owned by another CTA: scaled O^T, [head][dim], into this CTA's outgoing slots
    int o = 0;
    for (int dt = 0; dt < 4 && ns > 1; ++dt) {
      if (dt % ns == rank) continue;
      float* stg = reinterpret_cast<float*>(Mg + o * AD_TILE_BYTES) + 32 * q + lane;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t v[32];
        if (n_ch > 0) {
          umma::tmem_ld32(tmem + lane_addr + AD_O_COL + 64 * dt + 32 * hf, v);
          umma::tmem_ld_wait();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] = 0u;
        }
#pragma unroll
        for (int x = 0; x < 32; ++x) stg[(32 * hf + x) * 128] = __uint_as_float(v[x]) * fr[32 * hf + x];
      }
      ++o;
    }
  }
  umma::fence_proxy_async();   // the outgoing tiles are read by the bulk copies below
  __syncthreads();
  if (ns > 1 && tid == 0) {
    int o = 0;
    for (int dt = 0; dt < 4; ++dt) {
      const int owner = dt % ns;
      if (owner == rank) continue;
      // in the owner's incoming slots: [index of this CTA among its sources][owned tile]
      const int src_idx = rank < owner ? rank : rank - 1;
      const int own_o = tiles_owned(owner, ns);
      const uint32_t off = uint32_t(4 - own_o + src_idx * own_o + dt / ns) * AD_TILE_BYTES;
      bulk_to_peer(map_rank(Mg + off, owner), Mg + o * AD_TILE_BYTES, AD_TILE_BYTES,
                   map_rank(&recv_bar, owner));
      ++o;
    }
  }
  // owned tiles: own O^T (TMEM) plus the other CTAs' tiles (received), bf16 out
  if (o_warp) {
    const bool okr = ns == 1 || umma::mbar_wait(&recv_bar, 0, &d_err_attn);
    for (int lt = 0; rank + lt * ns < 4 && okr; ++lt) {
      const int dt = rank + lt * ns;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.out) + size_t(row) * NH * 512 +
                            dt * 128 + 32 * q + lane;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t v[32];
        if (n_ch > 0) {
          umma::tmem_ld32(tmem + lane_addr + AD_O_COL + 64 * dt + 32 * hf, v);
          umma::tmem_ld_wait();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] = 0u;
        }
        float acc[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) acc[x] = __uint_as_float(v[x]) * fr[32 * hf + x];
        for (int si = 0; si < ns - 1; ++si) {
          const float* in = reinterpret_cast<const float*>(Mg + (n_out + si * n_own + lt) * AD_TILE_BYTES) +
                            (32 * hf) * 128 + 32 * q + lane;
          float w[32];
#pragma unroll
          for (int x = 0; x < 32; ++x) w[x] = in[x * 128];
#pragma unroll
          for (int x = 0; x < 32; ++x) acc[x] += w[x];
        }
        if (H64) {
#pragma unroll
          for (int x = 0; x < 32; ++x) orow[(32 * hf + x) * 512] = __float2bfloat16_rn(acc[x]);
        } else {   // heads past H are not written
#pragma unroll
          for (int x = 0; x < 32; ++x)
            if (32 * hf + x < NH) orow[(32 * hf + x) * 512] = __float2bfloat16_rn(acc[x]);
        }
      }
    }
  }
  umma::fence_before();
  cluster.sync();   // no CTA leaves while a peer may still read or write its shared memory
  umma::fence_after();
  if (warp == 0) umma::tmem_free(tmem, 512);
}

// ---------------------------------------------------------------- persistent attention rows
// For calls with one CTA per query row (many rows: prefill, large batches) and bf16 rows: one
// CTA per SM walks rows blockIdx.x, blockIdx.x + gridDim.x, ... with the chunk pipeline of
// attn_decode_kernel, its chunk counter running on across rows, so that the next row's gathers,
// queries and score products proceed while the softmax warps write the current row's output.
// Window rows are gathered by the copy warps like the selected entries.  The queries of row
// j + 1 are loaded once the score products of row j have read its queries (q_free); the next
// row's first P V overwrites O^T only after the softmax warps have read it out (its
// probabilities are written after that row's output).
struct RowShape {
  int b, nw, n_wch, n_ch;
  long long t, lo;
};
__device__ __forceinline__ RowShape row_shape(const AttnArgs& a, int row) {
  RowShape r;
  r.b = row / a.Tq;
  r.t = (long long)a.q_pos0 + row % a.Tq;
  r.lo = r.t - a.window + 1 > 0 ? r.t - a.window + 1 : 0;
  r.nw = int(r.t - r.lo + 1);
  r.n_wch = (r.nw + AD_CH - 1) / AD_CH;
  r.n_ch = r.n_wch + (a.k + AD_CH - 1) / AD_CH;
  return r;
}

template <bool H64>
__global__ void __launch_bounds__(AD_T, 1) attn_rows_kernel(AttnArgs a, const __grid_constant__ CUtensorMap q_map) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* KV = base;                                   // 2 slots x 64 rows
  uint8_t* Qs = base + AD_SLOTS * AD_SLOT_BYTES;        // the row's queries
  uint8_t* Ps = Qs + AD_Q_BYTES;                        // 2 x P
  __shared__ int sidx[CSA2_MAX_TOPK];
  __shared__ const uint16_t* row_src[AD_SLOTS][AD_CH];
  __shared__ unsigned long long row_mask[AD_SLOTS];
  __shared__ __align__(8) uint64_t kv_full[AD_SLOTS], kv_empty[AD_SLOTS];
  __shared__ __align__(8) uint64_t s_full[2], s_empty[2], p_full[2], o_ready, q_full, q_free;
  __shared__ uint32_t tmem_slot;
  __shared__ float fac[64];
  const int NH = H64 ? 64 : a.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float scale_log2 = a.scale * 1.4426950408889634f;
  const int n_rows = a.rows > int(blockIdx.x) ? (a.rows - int(blockIdx.x) + int(gridDim.x) - 1) / int(gridDim.x) : 0;

  if (tid == 0) {
    for (int s = 0; s < AD_SLOTS; ++s) {
      umma::mbar_init(&kv_full[s], 1);
      umma::mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      umma::mbar_init(&s_full[s], 1);
      umma::mbar_init(&s_empty[s], 4);
      umma::mbar_init(&p_full[s], 4);
    }
    umma::mbar_init(&o_ready, 1);
    umma::mbar_init(&q_full, 1);
    umma::mbar_init(&q_free, 1);
    umma::mbar_fence_init();
  }
  if (warp == 0) umma::tmem_alloc(&tmem_slot, 512);
  if (!H64) {   // query rows H..63 of every plane are zero (the TMA fills rows 0..H-1)
    const int zb = (64 - a.H) * 128 / 16;   // (a.H < 64 here)
    for (int u = tid; u < 8 * zb; u += AD_T)
      *reinterpret_cast<uint4*>(Qs + (u / zb) * AD_PLANE + a.H * 128 + (u % zb) * 16) = make_uint4(0, 0, 0, 0);
    umma::fence_proxy_async();
  }
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;

  if (warp < 4) {
    // ---------------- copy warps: group g fills the chunks of slot g, global chunk g, g + 2, ...
    const int grp = warp >> 1, gt = tid & 63, gw = warp & 1;
    uint8_t* dst = KV + grp * AD_SLOT_BYTES;
    long long g_base = 0;   // global index of the row's first chunk
    for (int jr = 0; jr < n_rows; ++jr) {
      const int row = int(blockIdx.x) + jr * int(gridDim.x);
      const RowShape rs = row_shape(a, row);
      // both groups are past the previous row's chunks (and agree on going on)
      if (!bar_and(BAR_COPY, 128, ok)) { ok = false; break; }
      for (int j = tid; j < a.k; j += 128) sidx[j] = a.topk[size_t(row) * a.k + j];
      named_bar(BAR_COPY, 128);
      for (int c = int((grp ^ int(g_base & 1)) & 1); c < rs.n_ch && ok; c += AD_SLOTS) {
        const long long g = g_base + c;
        const int s = grp;
        const bool win = c < rs.n_wch;
        const int j = win ? c * AD_CH + gt : (c - rs.n_wch) * AD_CH + gt;
        int okr = 0;
        const uint16_t* src = nullptr;
        if (win) {
          if (j < rs.nw) {
            okr = 1;
            src = a.swa + (size_t(rs.b) * a.S + size_t(rs.lo + j - a.swa_pos0)) * 512;
          }
        } else if (j < a.k) {
          const int e = sidx[j];
          if (e >= a.n_entries) atomicOr(&d_err_attn, ERR_BOUNDS);
          if (e >= 0 && e < a.n_entries) {
            okr = 1;
            src = a.kv + (size_t(rs.b) * a.n_cap + e) * 512;
          }
        }
        const bool okw = g < AD_SLOTS || umma::mbar_wait(&kv_empty[s], ((g >> 1) - 1) & 1, &d_err_attn);
        {
          const unsigned m0 = __ballot_sync(0xffffffffu, okr);
          if (okw) {
            row_src[s][gt] = src;
            if (lane == 0) reinterpret_cast<unsigned*>(&row_mask[s])[gw] = m0;
          }
        }
        if (!bar_and(BAR_GROUP + grp, 64, okw)) { ok = false; break; }
#pragma unroll 1
        for (int r0 = 0; r0 < AD_CH; r0 += 8) {
          const uint16_t* sp[8];
#pragma unroll
          for (int u2 = 0; u2 < 8; ++u2) sp[u2] = row_src[s][r0 + u2];
#pragma unroll
          for (int u2 = 0; u2 < 8; ++u2)
            umma::cp_async16(dst + plane_off(r0 + u2, gt * 8), sp[u2] ? sp[u2] + gt * 8 : a.q,
                             sp[u2] ? 16u : 0u);
        }
        umma::cp_async_commit();
        umma::cp_async_wait_all();
        umma::fence_proxy_async();
        named_bar(BAR_GROUP + grp, 64);
        if (gt == 0) umma::mbar_arrive(&kv_full[s]);
      }
      g_base += rs.n_ch;
    }
  } else if (warp < 8) {
    // ---------------- softmax warps (as attn_decode_kernel), then each row's output
    const int q = warp & 3, h = 16 * q + (lane & 15);
    const bool head_lane = lane < 16;
    const int half = lane >> 4;
    const uint32_t lane_addr = uint32_t(32 * q) << 16;
    long long g_base = 0;
    for (int jr = 0; jr < n_rows && ok; ++jr) {
      const int row = int(blockIdx.x) + jr * int(gridDim.x);
      const RowShape rs = row_shape(a, row);
      float m_used = -INFINITY, l = 0.f, le = 0.f;
      for (int c = 0; c < rs.n_ch && ok; ++c) {
        const long long g = g_base + c;
        const int s = int(g & 1);
        const bool okc = __all_sync(0xffffffffu, umma::mbar_wait(&s_full[s], (g >> 1) & 1, &d_err_attn));
        if (!bar_and(BAR_SOFTMAX, 128, okc)) { ok = false; break; }
        umma::fence_after();
        float sv[AD_HALF];
        {
          uint32_t v0[32], v1[32];
          umma::tmem_ld32(tmem + lane_addr + AD_S_COL + 64 * s, v0);
          umma::tmem_ld32(tmem + lane_addr + AD_S_COL + 64 * s + 32, v1);
          umma::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < AD_HALF; ++j) {
            const float moved = __shfl_sync(0xffffffffu, __uint_as_float(v1[j]), lane & 15);
            sv[j] = half ? moved : __uint_as_float(v0[j]);
          }
        }
        umma::fence_before();
        __syncwarp();
        if (lane == 0) umma::mbar_arrive(&s_empty[s]);
        const unsigned mask = unsigned(row_mask[s] >> (half * AD_HALF));
        float cmx[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) cmx[x] = -INFINITY;
#pragma unroll
        for (int j = 0; j < AD_HALF; ++j) {
          sv[j] = ((mask >> j) & 1u) ? sv[j] * scale_log2 : -INFINITY;
          cmx[j & 7] = fmaxf(cmx[j & 7], sv[j]);
        }
        float cm = fmaxf(fmaxf(fmaxf(cmx[0], cmx[1]), fmaxf(cmx[2], cmx[3])),
                         fmaxf(fmaxf(cmx[4], cmx[5]), fmaxf(cmx[6], cmx[7])));
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
        float f = 1.f;
        if (cm > m_used + AD_LAZY || (m_used == -INFINITY && cm != -INFINITY)) {
          f = m_used == -INFINITY ? 0.f : exp2f(m_used - cm);
          m_used = cm;
          l *= f;
          le *= f;
        }
        float psx[4], pex[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) psx[x] = pex[x] = 0.f;
        uint32_t pk[AD_HALF / 2];
        const float msub = m_used == -INFINITY ? INFINITY : m_used;
#pragma unroll
        for (int j = 0; j < AD_HALF; j += 2) {
          const float p0 = fast_exp2(sv[j] - msub), p1 = fast_exp2(sv[j + 1] - msub);
          const __nv_bfloat162 v2 = __floats2bfloat162_rn(p0, p1);
          pk[j >> 1] = *reinterpret_cast<const uint32_t*>(&v2);
          const float2 r2 = __bfloat1622float2(v2);
          psx[(j >> 1) & 3] += r2.x + r2.y;
          pex[(j >> 1) & 3] += p0 + p1;
        }
        l += (psx[0] + psx[1]) + (psx[2] + psx[3]);
        le += (pex[0] + pex[1]) + (pex[2] + pex[3]);
        const bool okp = g < 2 || umma::mbar_wait(&kv_empty[s], ((g - 2) >> 1) & 1, &d_err_attn);
        if (!bar_and(BAR_SOFTMAX, 128, okp)) { ok = false; break; }
        uint8_t* pb = Ps + s * AD_P_BYTES + (h >> 3) * AD_P_SBO + (h & 7) * 16;
#pragma unroll
        for (int c4 = 0; c4 < AD_HALF / 8; ++c4) {
          const int kc = half * (AD_HALF / 8) + c4;
          *reinterpret_cast<uint4*>(pb + kc * 128) =
              make_uint4(pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
        }
        const bool need = head_lane && f != 1.f && c > 0;
        if (head_lane) fac[h] = need ? f : 1.f;
        if (bar_or(BAR_SOFTMAX, 128, need)) {
          const bool okr = __all_sync(0xffffffffu,
                                      umma::mbar_wait(&kv_empty[(g - 1) & 1], ((g - 1) >> 1) & 1, &d_err_attn));
          if (!bar_and(BAR_SOFTMAX, 128, okr)) { ok = false; break; }
          umma::fence_after();
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {
            float fr[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) fr[x] = fac[32 * hf + x];
#pragma unroll 1
            for (int dt = 0; dt < 4; ++dt) {
              uint32_t o[32];
              const uint32_t addr = tmem + lane_addr + AD_O_COL + 64 * dt + 32 * hf;
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
      if (!ok) break;
      // ---------------- the row's output: O^T (TMEM) / L per head, bf16
      const float l_fin = l + __shfl_xor_sync(0xffffffffu, l, 16);
      const float e_fin = le + __shfl_xor_sync(0xffffffffu, le, 16);
      // the row's products are complete; every warp is past its rescales (fac reused)
      ok = bar_and(BAR_SOFTMAX, 128, umma::mbar_wait(&o_ready, jr & 1, &d_err_attn));
      if (!ok) break;
      umma::fence_after();
      if (head_lane) {
        const float sk = a.sink && h < NH ? a.sink[h] * 1.4426950408889634f : -INFINITY;
        const float M = fmaxf(sk, m_used);
        float L = a.sink ? exp2f(sk - M) : 0.f, Le = L;
        if (l_fin > 0.f) {
          const float gm = exp2f(m_used - M);
          L += l_fin * gm;
          Le += e_fin * gm;
        }
        fac[h] = l_fin > 0.f ? exp2f(m_used - M) / L : 0.f;
        if (a.lse && h < NH) a.lse[size_t(row) * NH + h] = (M + log2f(Le)) * 0.6931471805599453f;
      }
      named_bar(BAR_SOFTMAX, 128);
      float fr[64];
#pragma unroll
      for (int x = 0; x < 64; ++x) fr[x] = fac[x];
      named_bar(BAR_SOFTMAX, 128);   // fac is free for the next row's rescales
#pragma unroll 1
      for (int dt = 0; dt < 4; ++dt) {
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.out) + size_t(row) * NH * 512 +
                              dt * 128 + 32 * q + lane;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t v[32];
          umma::tmem_ld32(tmem + lane_addr + AD_O_COL + 64 * dt + 32 * hf, v);
          umma::tmem_ld_wait();
          if (H64) {
#pragma unroll
            for (int x = 0; x < 32; ++x)
              orow[(32 * hf + x) * 512] = __float2bfloat16_rn(__uint_as_float(v[x]) * fr[32 * hf + x]);
          } else {
#pragma unroll
            for (int x = 0; x < 32; ++x)
              if (32 * hf + x < NH)
                orow[(32 * hf + x) * 512] = __float2bfloat16_rn(__uint_as_float(v[x]) * fr[32 * hf + x]);
          }
        }
      }
      g_base += rs.n_ch;
    }
  } else if (warp == 8 && lane == 0) {
    // ---------------- TMA (queries) and MMA issuer over all rows' chunks
    constexpr uint32_t idesc_s = umma::idesc_f16(64, AD_CH, 1, 0, 0);
    constexpr uint32_t idesc_o = umma::idesc_f16(128, 64, 1, 1, 0);
    const uint32_t kv0 = umma::smem_u32(KV), q0 = umma::smem_u32(Qs), p0 = umma::smem_u32(Ps);
    auto load_q = [&](int jr) {
      const int row = int(blockIdx.x) + jr * int(gridDim.x);
      mbar_expect_tx(&q_full, uint32_t(NH) * 1024u);
#pragma unroll 1
      for (int j = 0; j < 8; ++j) tma_load_2d(Qs + j * AD_PLANE, &q_map, 64 * j, row * NH, &q_full);
    };
    auto issue_s = [&](long long g) {
      const int s = int(g & 1);
      umma::fence_after();
      const uint64_t da0 = umma::desc_sw128(q0, 16, 1024);
      const uint64_t db0 = umma::desc_sw128(kv0 + s * AD_SLOT_BYTES, 16, 1024);
#pragma unroll
      for (int ks = 0; ks < 32; ++ks) {
        const uint32_t off = uint32_t(((ks >> 2) * AD_PLANE + (ks & 3) * 32) >> 4);
        umma::mma_f16(tmem + AD_S_COL + 64 * s, da0 + off, db0 + off, idesc_s, ks > 0 ? 1u : 0u);
      }
      umma::commit(&s_full[s]);
    };
    auto issue_pv = [&](long long g, bool first) {
      const int s = int(g & 1);
      umma::fence_after();
      const uint64_t pa0 = umma::desc_sw128(kv0 + s * AD_SLOT_BYTES, AD_PLANE, 1024);
      const uint64_t pb0 = desc_noswz(p0 + s * AD_P_BYTES, 128, AD_P_SBO);
#pragma unroll
      for (int kk = 0; kk < AD_CH / 16; ++kk)
#pragma unroll
        for (int dt = 0; dt < 4; ++dt)
          umma::mma_f16(tmem + AD_O_COL + 64 * dt, pa0 + uint32_t(((2 * dt) * AD_PLANE + kk * 2048) >> 4),
                        pb0 + uint32_t((kk * 256) >> 4), idesc_o, (!first || kk > 0) ? 1u : 0u);
      umma::commit(&kv_empty[s]);
    };
    if (n_rows > 0) load_q(0);
    int js = 0, cs = 0, jp = 0, cp = 0;        // next S and next P V: row (of this CTA), chunk
    long long gs = 0, gp = 0;                  // their global chunk indices
    int nch_s = n_rows > 0 ? row_shape(a, int(blockIdx.x)).n_ch : 0, nch_p = nch_s;
    int q_wait = -1;                           // row whose queries wait for the previous row's S
    uint32_t idle = 0;
    while (jp < n_rows) {
      if (q_wait >= 0 && umma::mbar_test(&q_free, (q_wait - 1) & 1)) {
        load_q(q_wait);
        q_wait = -1;
        idle = 0;
      }
      if (js < n_rows && gs <= gp + 1) {
        const int s = int(gs & 1);
        if (umma::mbar_test(&kv_full[s], (gs >> 1) & 1) && (cs != 0 || umma::mbar_test(&q_full, js & 1)) &&
            (gs < 2 || umma::mbar_test(&s_empty[s], ((gs >> 1) - 1) & 1))) {
          issue_s(gs);
          ++gs;
          if (++cs == nch_s) {   // the row's queries are read once these products complete
            umma::commit(&q_free);
            if (++js < n_rows) {
              q_wait = js;
              nch_s = row_shape(a, int(blockIdx.x) + js * int(gridDim.x)).n_ch;
            }
            cs = 0;
          }
          idle = 0;
          continue;
        }
      }
      if (gp < gs && umma::mbar_test(&p_full[gp & 1], (gp >> 1) & 1)) {
        issue_pv(gp, cp == 0);
        ++gp;
        if (++cp == nch_p) {
          umma::commit(&o_ready);
          if (++jp < n_rows) nch_p = row_shape(a, int(blockIdx.x) + jp * int(gridDim.x)).n_ch;
          cp = 0;
        }
        idle = 0;
        continue;
      }
      if (++idle > (1u << 26)) { atomicOr(&d_err_attn, ERR_TIMEOUT); break; }
    }
  }
  umma::fence_before();
  __syncthreads();
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
  // the tensor-core kernel takes up to 64 heads in multiples of 8 (its query tile has 64 rows,
  // loaded by TMA 8-row atoms; rows past H are zero); other head counts take the SIMT kernel
  const bool tc = H <= 64 && H % 8 == 0;
  if ((fp4 || fp8w) && !tc)
    return fail(CSA2_ERR_UNSUPPORTED, "sparse_attn: quantised entries or rows need H a multiple of 8 up to 64 (got %d)", H);
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
  if (tc) {
    // tensor-core path: a cluster of n_split CTAs per row, partial results merged through
    // distributed shared memory; queries (and bf16 window rows) through tensor maps
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
      e0 = cudaFuncSetAttribute(attn_decode_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(AD_SMEM));
      if (e0 == cudaSuccess)
        e0 = cudaFuncSetAttribute(attn_decode_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(AD_SMEM));
      if (e0 == cudaSuccess)
        e0 = cudaFuncSetAttribute(attn_decode_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(AD_SMEM));
      if (e0 == cudaSuccess)
        e0 = cudaFuncSetAttribute(attn_decode_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(AD_SMEM));
      if (e0 == cudaSuccess)
        e0 = cudaFuncSetAttribute(attn_rows_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(AD_SMEM));
      if (e0 == cudaSuccess)
        e0 = cudaFuncSetAttribute(attn_rows_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(AD_SMEM));
      if (e0 == cudaSuccess) e0 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e0 != cudaSuccess) return cuda_fail(e0, "sparse_attn: attributes");
      sms_cache[dev].store(sms, std::memory_order_release);
    }
    if (rows * H > (1ll << 31) - 1) return fail(CSA2_ERR_UNSUPPORTED, "sparse_attn: too many query rows");
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return fail(CSA2_ERR_CUDA, "sparse_attn: cuTensorMapEncodeTiled not available");
    // queries: [rows * H heads][512 dims] bf16, one box = H heads x 64 dims (one plane's
    // first H rows)
    CUtensorMap q_map, swa_map;
    {
      const cuuint64_t dims[2] = {512, cuuint64_t(rows * H)};
      const cuuint64_t strides[1] = {1024};
      const cuuint32_t box[2] = {64, cuuint32_t(H)};
      const cuuint32_t estr[2] = {1, 1};
      if (enc(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return fail(CSA2_ERR_CUDA, "sparse_attn: query tensor map");
    }
    // bf16 window rows: [B][rows up to the last query's position][512 dims]; rows past the
    // last query are outside the map and read as zeros
    int win_tma = 0;
    swa_map = q_map;   // (unused unless the window rows are bf16)
    if (swa_kv) {
      const long long valid = std::min<long long>(S, (long long)q_pos0 + Tq - swa_pos0);
      const cuuint64_t dims[3] = {512, cuuint64_t(valid), cuuint64_t(B)};
      const cuuint64_t strides[2] = {1024, cuuint64_t(S) * 1024};
      const cuuint32_t box[3] = {64, 64, 1};
      const cuuint32_t estr[3] = {1, 1, 1};
      if (enc(&swa_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(swa_kv), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return fail(CSA2_ERR_CUDA, "sparse_attn: window tensor map");
      win_tma = 1;
    }
    // CTAs per row: all CTAs in one wave, and the estimated time of a CTA's chunks (about
    // 1.4 us each) plus the cluster merge (about 2 us) the smallest
    const int n_ch_max = ceil_div(k, AD_CH) + ceil_div(window, AD_CH);
    const int n_fit = std::max(1, std::min(int(sms / rows), AD_MAX_SPLIT));
    int n_split = 1;
    for (int n = 2; n <= n_fit; ++n) {
      const int t_n = 7 * ceil_div(n_ch_max, n) + 10, t_best = 7 * ceil_div(n_ch_max, n_split) + (n_split > 1 ? 10 : 0);
      if (t_n < t_best) n_split = n;
    }
    if (rows * n_split > (1ll << 31) - 1) return fail(CSA2_ERR_UNSUPPORTED, "sparse_attn: too many rows");
    AttnDecodeArgs da{aa, n_split, win_tma};
    const dim3 grid(unsigned(rows * n_split), 1, 1), block(AD_T, 1, 1);
    const bool q8 = fp4 || fp8w;
    if (n_split == 1 && !q8 && rows > sms) {
      // more rows than SMs, bf16 rows: one persistent CTA per SM walks its rows
      const dim3 pgrid(unsigned(sms), 1, 1);
      e0 = H == 64 ? launch_k(attn_rows_kernel<true>, pgrid, block, AD_SMEM, st, 1u, aa, q_map)
                   : launch_k(attn_rows_kernel<false>, pgrid, block, AD_SMEM, st, 1u, aa, q_map);
    } else if (H == 64)
      e0 = q8 ? launch_k(attn_decode_kernel<true, true>, grid, block, AD_SMEM, st, unsigned(n_split), da, q_map, swa_map)
              : launch_k(attn_decode_kernel<false, true>, grid, block, AD_SMEM, st, unsigned(n_split), da, q_map, swa_map);
    else
      e0 = q8 ? launch_k(attn_decode_kernel<true, false>, grid, block, AD_SMEM, st, unsigned(n_split), da, q_map, swa_map)
              : launch_k(attn_decode_kernel<false, false>, grid, block, AD_SMEM, st, unsigned(n_split), da, q_map, swa_map);
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
