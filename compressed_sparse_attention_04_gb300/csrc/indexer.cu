// Stage 3: lightning-indexer scores, causal top-k, HSI candidate pools.
//
// [P1] "DeepSeek-V4.1 模型结构（2）：序列维度（中），CSA2 的三种模式" (blog.javazero.top),
//      §indexer K 改由 main KV 投影: score of entry s for token t is the sum over the 32
//      indexer heads of the head weight times ReLU(q_{t,j} . k_s), 128 dims per head;
//      512 entries are kept per query.
// [P2] "DeepSeek v4.1 Flash技术剖析——架构篇" (myhz0606.com), §Indexer (causally visible
//      set), §CSA2-ReIndex (block max scores, top blocks form the pool, the newest
//      visible block is forced in, non-pool entries scored -inf).
// [P3] "DeepSeek-V4.1-Flash：把百万 Token 的记忆，压缩成一套分级缓存" (junki.cn), §五 HSI.
//
// Kernels
//   score_kernel   one CTA per (query row, chunk of 1024 entries or pool slots): the CTA
//                  quantises its query to FP4 (same rule as the keys), then each thread
//                  scores one entry per pass: 32 heads x 4 blocks of 32 dims; the block
//                  partial sums are exact in float32 and are scaled once by the key scale.
//   score_fp4_kernel  tensor-core version of score_kernel (block <= 128): keys on M = 128,
//                  the 32 heads on N, K = 128, block-scaled FP4 MMA.  Producer warps copy
//                  the keys' packed codes straight into the operand image and put the block
//                  scales into TMEM; one thread issues two MMAs per tile into a
//                  double-buffered TMEM accumulator; epilogue warps apply ReLU and the head
//                  weights.  The 16-value block products are exact; only float32
//                  accumulation rounds.
//   topk_kernel    one CTA per query row: radix select (select.cuh).
//   hsi_kernel     one CTA per query row: top-nb blocks with the newest block forced.
#include <cuda.h>
#include <algorithm>
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "select.cuh"
#include "umma.cuh"

CSA2_DEFINE_ERR_WORD(d_err_indexer)

namespace csa2 {
namespace {

constexpr int SC_T = 256;       // threads per scoring CTA
constexpr int SC_CHUNK = 1024;  // entries (or pool slots) per scoring CTA

struct ScoreArgs {
  const uint16_t* q_idx;   // [rows, 32, 128]
  const float* w;          // [rows, 32]
  int rows, Tq, q_pos0;
  const uint8_t* codes;    // [B, n_cap, 64]
  const uint8_t* scales;   // [B, n_cap, 4]
  int n_cap, n_entries, m;
  const int32_t* cand;     // [rows, nb] or null
  int nb, blk, n_blocks;   // n_blocks = ceil(n_entries / blk)
  float* scores;           // [rows, row_len]
  int row_len;
  float* blockmax;         // [rows, n_blocks] or null
  int n_chunks;
  int use_tma;             // codes through the tensor map (n_cap % 64 == 0, pool blk == 64)
  const uint8_t* qprep;    // [rows][SU_QROW_BYTES] FP4 query images (tensor-core path)
  const int* prefix;       // [Tq + 1] exclusive prefix of the steps per query index
  long long total_steps;   // B * prefix[Tq]
  float* bm64;             // [rows][nb64] maxima of 64-key blocks for the top-k threshold, or null
  int nb64;
  uint32_t wait_limit;     // (tensor-core decode scorer) polls per device wait
  int stall;               // (tensor-core decode scorer) the copy thread first waits on a
                           // barrier that nothing completes, so that every wait runs out
};

__global__ void __launch_bounds__(SC_T) score_kernel(ScoreArgs a) {
  pdl_wait();
  __shared__ __align__(16) float qh[32][128];
  __shared__ float wsh[32];
  __shared__ float sbuf[SC_T];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x / a.n_chunks, chunk = blockIdx.x % a.n_chunks;
  const int b = row / a.Tq, i = row % a.Tq;
  const long long t = (long long)a.q_pos0 + i;
  const int n_vis = n_visible(t, a.m, a.n_entries);
  const int c0 = chunk * SC_CHUNK;
  const bool pool = a.cand != nullptr;
  const int limit = pool ? a.row_len : n_vis;
  if (c0 >= limit && a.blockmax == nullptr) return;   // uniform

  // FP4-quantise the query: warp w handles 16 (head, block) pairs, lane = element
  const uint16_t* qrow = a.q_idx + size_t(row) * 32 * 128;
  for (int pb = warp; pb < 128; pb += SC_T / 32) {
    const int h = pb >> 2, blk4 = pb & 3;
    const float v = bf16_to_f32(qrow[h * 128 + blk4 * 32 + lane]);
    uint32_t sb;
    const uint32_t code = fp4_quant_lane(v, sb);
    qh[h][blk4 * 32 + lane] = e2m1_value(code) * e4m3_value(sb);
  }
  if (tid < 32) wsh[tid] = a.w[size_t(row) * 32 + tid];
  __syncthreads();

  const size_t cache_row0 = size_t(b) * a.n_cap;
  for (int it = 0; it < SC_CHUNK / SC_T; ++it) {
    const int p = c0 + it * SC_T + tid;
    float score = -INFINITY;
    long long e = -1;
    if (p < limit) {
      if (pool) {
        const int cb = a.cand[size_t(row) * a.nb + p / a.blk];
        if (cb >= 0) {
          if (cb >= a.n_blocks) {
            atomicOr(&d_err_indexer, ERR_BOUNDS);
          } else {
            const long long ee = (long long)cb * a.blk + (p % a.blk);
            if (ee < n_vis) e = ee;
          }
        }
      } else {
        e = p;
      }
    }
    if (e >= 0) {
      const uint8_t* crow = a.codes + (cache_row0 + size_t(e)) * 64;
      const uint32_t sc4 = *reinterpret_cast<const uint32_t*>(a.scales + (cache_row0 + size_t(e)) * 4);
      float d[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) d[j] = 0.f;
#pragma unroll 1
      for (int kb = 0; kb < 4; ++kb) {
        const uint4 cv = *reinterpret_cast<const uint4*>(crow + kb * 16);
        const uint32_t wds[4] = {cv.x, cv.y, cv.z, cv.w};
        float kv[32];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int nn = 0; nn < 8; ++nn) kv[u * 8 + nn] = e2m1_value((wds[u] >> (4 * nn)) & 0xFu);
        const float sk = e4m3_value((sc4 >> (8 * kb)) & 0xFFu);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float4* qv = reinterpret_cast<const float4*>(&qh[j][kb * 32]);
          float part = 0.f;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float4 q4 = qv[u];
            part = fmaf(q4.x, kv[4 * u + 0], part);
            part = fmaf(q4.y, kv[4 * u + 1], part);
            part = fmaf(q4.z, kv[4 * u + 2], part);
            part = fmaf(q4.w, kv[4 * u + 3], part);
          }
          d[j] = fmaf(part, sk, d[j]);
        }
      }
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) s = fmaf(wsh[j], fmaxf(d[j], 0.f), s);
      score = s;
    }
    if (p < a.row_len && (pool || p < n_vis)) a.scores[size_t(row) * a.row_len + p] = score;
    if (a.blockmax) {
      sbuf[tid] = score;
      __syncthreads();
      const int per = SC_T / a.blk;   // blocks in this pass (blk <= 256, power of two)
      if (tid < per) {
        float mx = -INFINITY;
        for (int u = 0; u < a.blk; ++u) mx = fmaxf(mx, sbuf[tid * a.blk + u]);
        const int bi = (c0 + it * SC_T) / a.blk + tid;
        if (bi < a.n_blocks) a.blockmax[size_t(row) * a.n_blocks + bi] = mx;
      }
      __syncthreads();
    }
  }
}


// ---------------------------------------------------------------- tensor-core scoring
// Block-scaled FP4 MMA (kind::mxf4nvf4, scale_vec::4X): the packed E2M1 key codes are the
// A operand as stored (128 keys x 64 bytes per tile, K-major, no swizzle: 8-row x 16-byte
// core matrices, LBO = 128, SBO = 512), the query's FP4 codes the B operand, and the
// E4M3 scales (one per 32 dims, given to the MMA once per 16) sit in TMEM in the
// replicated chunk layout: word g of lane i holds the four block scales of row i + 32 g.
// The MMA yields sum_blocks s_q s_k sum(e2m1 products) per (key, head) = q_hat . k_hat.
constexpr int SU_TILE = 128;                 // keys per MMA tile (M)
constexpr int SU_STEP = 256;                 // keys per pipeline step: two MMA tiles
constexpr int SU_STAGES = 6;                 // code / scale ring (in steps)
constexpr int SU_ND = 2;                     // TMEM accumulator buffers (in steps)
constexpr int SU_T = 320;                    // 4 producer + 4 epilogue + 1 MMA + 1 copy warp
constexpr uint32_t SU_A_BYTES = SU_TILE * 64;          // 8 KB of codes per tile
constexpr uint32_t SU_STAGE_BYTES = 2 * SU_A_BYTES;    // 16 KB of codes per step
constexpr uint32_t SU_Q_BYTES = 32 * 64;               // 2 KB of query codes
constexpr uint32_t SU_QROW_BYTES = SU_Q_BYTES + 128;   // + 32 per-head scale words
// code / scale ring, two query buffers (rows change inside a CTA's step range), alignment
constexpr uint32_t SU_SMEM = SU_STAGES * (SU_STAGE_BYTES + SU_STEP * 4) + 2 * SU_QROW_BYTES + 1024;
constexpr uint32_t SU_TMEM_COLS = 256;       // D 2 x 64 | SFA 6 x 16 | SFB 2 x 8
constexpr uint32_t SU_SFA_COL = 128, SU_SFB_COL = 224;
constexpr uint32_t SU_IDESC = (1u << 7) | (1u << 10) | ((32u >> 3) << 17) | ((128u >> 4) << 24);

// byte offset of 16-byte chunk c (0..3) of row r in the no-swizzle K-major FP4 image
__device__ __forceinline__ uint32_t fp4_chunk_off(int r, int c) {
  return uint32_t((r >> 3) * 512 + c * 128 + (r & 7) * 16);
}
__device__ __forceinline__ uint64_t desc_noswz(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t(128u >> 4) << 16;   // LBO: next 16-byte column of core matrices (K)
  d |= uint64_t(512u >> 4) << 32;   // SBO: next group of 8 rows (M / N)
  d |= uint64_t(1) << 46;
  return d;
}
__device__ __forceinline__ void mma_fp4(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t sfa,
                                        uint32_t sfb, uint32_t accumulate, uint32_t idesc = SU_IDESC) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      :: "r"(tmem_d), "l"(da), "l"(db), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate));
}
// per-16 scale words for the two K = 64 halves from four per-32 E4M3 bytes: (s0 s0 s1 s1),
// (s2 s2 s3 s3)
__device__ __forceinline__ uint32_t sf_lo(uint32_t s4) { return __byte_perm(s4, 0u, 0x1100); }
__device__ __forceinline__ uint32_t sf_hi(uint32_t s4) { return __byte_perm(s4, 0u, 0x3322); }

// Placement of the 256 keys of a step in the two 128-row MMA tiles: step key 64 q + l
// (l < 32) goes to row 32 q + l of tile 0, step key 64 q + 32 + l to row 32 q + l of
// tile 1.  Epilogue warp q (TMEM lanes 32 q ..) then holds step keys 64 q .. 64 q + 63,
// a whole 64-key block, so block maxima need no exchange between warps.
__device__ __forceinline__ void step_slot(int kk, int& tile, int& r) {
  const int q = kk >> 6, w = kk & 63;
  tile = w >> 5;
  r = q * 32 + (w & 31);
}

__device__ __forceinline__ uint64_t desc_sw64(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t(512u >> 4) << 32;   // SBO: next group of 8 rows of 64 bytes
  d |= uint64_t(1) << 46;
  d |= uint64_t(4) << 61;           // SWIZZLE_64B
  return d;
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            int c3, void* mbar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5}], [%6];"
      :: "r"(umma::smem_u32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
         "r"(umma::smem_u32(mbar)) : "memory");
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, void* mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(umma::smem_u32(dst)), "l"(src), "r"(bytes), "r"(umma::smem_u32(mbar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(void* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
               :: "r"(umma::smem_u32(bar)), "r"(bytes) : "memory");
}

// ---- persistent schedule: the steps of all rows, in row order, split evenly over the CTAs.
// A row (query) has ceil(span / SU_STEP) steps, span = the pool length, or the visible
// entries, or (when block maxima are produced) the whole row.  The steps of a row depend
// only on the query index i, so one prefix table over i serves all sequences.
__host__ __device__ inline int row_steps(int i, int q_pos0, int m, int n_entries, int row_len,
                                         bool pool, bool blockmax) {
  const int limit = pool ? row_len : n_visible((long long)q_pos0 + i, m, n_entries);
  const int span = blockmax ? row_len : limit;
  return (span + SU_STEP - 1) / SU_STEP;
}

// Walks the (sequence, query index, step) triples from a flat step number.
struct StepCursor {
  int b, i, st, n, k;   // sequence, query index, step within the row, steps in the row,
                        // rows entered so far by this CTA minus one
  __device__ void init(const ScoreArgs& a, long long s) {
    const int T = a.prefix[a.Tq];
    b = int(s / T);
    const int r = int(s % T);
    int lo = 0, hi = a.Tq - 1;   // largest i with prefix[i] <= r (that row has steps)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.prefix[mid] <= r) lo = mid; else hi = mid - 1;
    }
    i = lo;
    st = r - a.prefix[i];
    n = a.prefix[i + 1] - a.prefix[i];
    k = 0;
  }
  // Advance one step; true when it enters a new row.  Only called while steps remain.
  __device__ bool next(const ScoreArgs& a) {
    if (++st < n) return false;
    do {
      if (++i == a.Tq) { i = 0; ++b; }
      n = a.prefix[i + 1] - a.prefix[i];
    } while (n == 0);
    st = 0;
    ++k;
    return true;
  }
  __device__ int row(const ScoreArgs& a) const { return b * a.Tq + i; }
};

// ---- prefill scoring (score_prefill_kernel below): PF_QG consecutive queries of a
// sequence share each 128-key tile, their 32 heads each side by side on the MMA's N.
constexpr int PF_QG = 4;                        // queries per group (N = 128)
constexpr int PF_TILE = 128;                    // keys per step (M)
constexpr int PF_STAGES = 8;                    // key ring
constexpr int PF_ND = 3;                        // TMEM accumulators (steps)
constexpr int PF_T = 704;                       // copy, MMA, 4 scale-factor and 16 epilogue warps
constexpr uint32_t PF_A_BYTES = PF_TILE * 64;   // 8 KB of codes per step
constexpr uint32_t PF_Q_IMG = PF_QG * SU_Q_BYTES;            // 8 KB of query codes per group
constexpr uint32_t PF_Q_SC = PF_QG * 128;                    // their scale words
constexpr uint32_t PF_SMEM = PF_STAGES * (PF_A_BYTES + PF_TILE * 4) + 2 * (PF_Q_IMG + PF_Q_SC) + 1024;
constexpr uint32_t PF_SFA_COL = 384, PF_SFB_COL = 448;       // D: 3 x 128 columns
constexpr uint32_t PF_IDESC = (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr int PF_MIN_TQ = 64;                   // calls with fewer queries keep the decode scorer

// One warp per (query row, head), grid-stride: the FP4 query as the MMA's B operand image
// (32 heads x 64 bytes, K-major, no swizzle) followed by its E4M3 block scales (4 bytes per
// head).  Lane l holds dims 4 l .. 4 l + 3, so lanes 8 b .. 8 b + 7 form 32-dim block b; the
// block's scale and codes follow the same rules as fp4_quant_lane.  CTA 0 also writes the
// step prefix table.
// Where q_prep writes a row's FP4 image and scale words (decode: image and scales of a row
// together, SU_QROW_BYTES apart; prefill: images 2 KB apart, scale words 128 B apart, so that
// the images of consecutive queries form one operand), and which step table it builds.
struct QPrepOut {
  uint8_t* img;
  uint32_t img_stride;
  uint8_t* sc;
  uint32_t sc_stride;
  int groups;   // prefill scorer: steps per group of PF_QG queries instead of per query
};

__global__ void __launch_bounds__(128) q_prep_kernel(ScoreArgs a, QPrepOut qo, int* prefix,
                                                     long long n_items) {
  pdl_wait();
  __shared__ int scan[32];
  const int tid = threadIdx.x, lane = tid & 31, blk = lane >> 3, l8 = lane & 7;
  // four items per warp and round, their loads issued together
  const long long stride = (long long)gridDim.x * 4;
  for (long long item0 = (long long)blockIdx.x * 4 + (tid >> 5); item0 < n_items; item0 += 4 * stride) {
    uint2 raws[4];
#pragma unroll
    for (int r4 = 0; r4 < 4; ++r4) {
      const long long it = min(item0 + r4 * stride, n_items - 1);
      raws[r4] = *reinterpret_cast<const uint2*>(a.q_idx + size_t(it >> 5) * 32 * 128 + int(it & 31) * 128 + 4 * lane);
    }
#pragma unroll
    for (int r4 = 0; r4 < 4; ++r4) {
      const long long item = item0 + r4 * stride;
      if (item >= n_items) break;   // uniform across the warp
      const long long row = item >> 5;
      const int h = int(item & 31);
      const uint2 raw = raws[r4];
      const float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                          __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
      float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
      const uint32_t sb = e4m3_rne_satfinite(__fdiv_rn(amax, 6.0f));
      // this lane's four codes: elements 4 l8 .. 4 l8 + 3 of the block = nibbles 4 (l8 & 1) ..
      // 4 (l8 & 1) + 3 of the block's word l8 / 2 (element 8 j + i in nibble i of word j)
      uint32_t part = 0u;
      if (sb != 0u) {
        const float sc = e4m3_value(sb);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float u = __fdiv_rn(v[e], sc);
          part |= (((__float_as_uint(u) >> 31) << 3) | e2m1_rne_mag(fabsf(u))) << (4 * e);
        }
      }
      const uint32_t word = (part << (16 * (l8 & 1))) | (__shfl_xor_sync(0xffffffffu, part, 1) << (16 * ((l8 & 1) ^ 1)));
      const uint32_t w1 = __shfl_sync(0xffffffffu, word, (lane & ~7) + 2);
      const uint32_t w2 = __shfl_sync(0xffffffffu, word, (lane & ~7) + 4);
      const uint32_t w3 = __shfl_sync(0xffffffffu, word, (lane & ~7) + 6);
      if (l8 == 0) {
        *reinterpret_cast<uint4*>(qo.img + size_t(row) * qo.img_stride + fp4_chunk_off(h, blk)) =
            make_uint4(word, w1, w2, w3);
        qo.sc[size_t(row) * qo.sc_stride + h * 4 + blk] = uint8_t(sb);
      }
    }
  }
  if (blockIdx.x == 0 && qo.groups) {
    // prefill: the 128-key steps of each group of PF_QG queries (the group's last query
    // sees the most entries)
    const int G = (a.Tq + PF_QG - 1) / PF_QG;
    const int per = (G + 127) / 128, g0 = tid * per, g1 = min(G, g0 + per);
    auto steps = [&](int g) {
      const int last = min(a.Tq - 1, PF_QG * g + PF_QG - 1);
      return (n_visible((long long)a.q_pos0 + last, a.m, a.n_entries) + PF_TILE - 1) / PF_TILE;
    };
    int mine = 0;
    for (int g = g0; g < g1; ++g) mine += steps(g);
    int tot;
    int run = block_excl_scan<128>(mine, scan, tot);
    for (int g = g0; g < g1; ++g) {
      prefix[g] = run;
      run += steps(g);
    }
    if (tid == 0) prefix[G] = tot;
  } else if (blockIdx.x == 0) {
    // thread t sums the steps of rows [t per, (t + 1) per), one block scan of the 128 sums,
    // then each thread writes its rows' offsets (one scan instead of Tq / 128 of them)
    const bool pool = a.cand != nullptr, bm = a.blockmax != nullptr;
    const int per = (a.Tq + 127) / 128, i0 = tid * per, i1 = min(a.Tq, i0 + per);
    int mine = 0;
    for (int i = i0; i < i1; ++i) mine += row_steps(i, a.q_pos0, a.m, a.n_entries, a.row_len, pool, bm);
    int tot;
    int run = block_excl_scan<128>(mine, scan, tot);
    for (int i = i0; i < i1; ++i) {
      prefix[i] = run;
      run += row_steps(i, a.q_pos0, a.m, a.n_entries, a.row_len, pool, bm);
    }
    if (tid == 0) prefix[a.Tq] = tot;
  }
}

__global__ void __launch_bounds__(SU_T, 2) score_fp4_kernel(ScoreArgs a, const __grid_constant__ CUtensorMap codes_map,
                                                          const __grid_constant__ CUtensorMap codes_map4) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* As = base;                                              // SU_STAGES x 2 tiles x 8 KB
  uint32_t* Ss = reinterpret_cast<uint32_t*>(base + SU_STAGES * SU_STAGE_BYTES);   // SU_STAGES x 256
  uint8_t* Qb = base + SU_STAGES * (SU_STAGE_BYTES + SU_STEP * 4);  // 2 x query image + scales
  __shared__ __align__(8) uint64_t a_empty[SU_STAGES], land[SU_STAGES], sf_ready[SU_STAGES];
  __shared__ __align__(8) uint64_t d_full[SU_ND], d_empty[SU_ND], q_empty[2], never;
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t polls = a.wait_limit;
  const long long S = a.total_steps;
  const long long s_begin = S * blockIdx.x / gridDim.x, s_end = S * (blockIdx.x + 1) / gridDim.x;
  const int L = int(s_end - s_begin);
  if (L <= 0) return;   // uniform
  const bool pool = a.cand != nullptr;

  if (tid == 0) {
    for (int s2 = 0; s2 < SU_STAGES; ++s2) {
      umma::mbar_init(&a_empty[s2], 1);
      // TMA: the copy thread's arrive with the byte count; otherwise also the producers'
      umma::mbar_init(&land[s2], a.use_tma ? 1 : 129);
      umma::mbar_init(&sf_ready[s2], 4);
    }
    for (int d = 0; d < SU_ND; ++d) {
      umma::mbar_init(&d_full[d], 1);
      umma::mbar_init(&d_empty[d], 4);
    }
    umma::mbar_init(&q_empty[0], 1);
    umma::mbar_init(&q_empty[1], 1);
    umma::mbar_init(&never, 1);
    umma::mbar_fence_init();
  }
  if (warp == 0) umma::tmem_alloc(&tmem_slot, SU_TMEM_COLS);
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp < 4) {
    // ---------------- producers: (without the tensor map) the codes and scale bytes by
    // cp.async; then this warp's quadrant of the scale factors into TMEM.
    const uint32_t lane_addr = uint32_t(warp * 32) << 16;
    StepCursor ci, cs;   // copy cursor (runs PF steps ahead), scale-factor cursor
    ci.init(a, s_begin);
    cs.init(a, s_begin);
    // 16-byte unit u = 4 * key + chunk of the step: consecutive threads copy consecutive
    // units, so a warp reads 512 contiguous bytes whenever the keys are contiguous.
    auto issue = [&](int g) {
      if (g < L) {
        if (g > 0) ci.next(a);
        const int s2 = g % SU_STAGES;
        if (g >= SU_STAGES &&
            !umma::mbar_wait(&a_empty[s2], ((g / SU_STAGES) - 1) & 1, &d_err_indexer, polls)) return false;
        const int row = ci.row(a);
        const int n_vis = n_visible((long long)a.q_pos0 + ci.i, a.m, a.n_entries);
        const int limit = pool ? a.row_len : n_vis;
        const size_t cache_row0 = size_t(ci.b) * a.n_cap;
        auto key_at = [&](int kk) -> long long {   // entry of step key kk (or -1)
          const int p = ci.st * SU_STEP + kk;
          if (p >= limit) return -1;
          if (!pool) return p;
          const int cb = a.cand[size_t(row) * a.nb + p / a.blk];
          if (cb < 0 || cb >= a.n_blocks) return -1;
          const long long ee = (long long)cb * a.blk + (p % a.blk);
          return ee < n_vis ? ee : -1;
        };
        uint8_t* dst = As + s2 * SU_STAGE_BYTES;
#pragma unroll
        for (int rep = 0; rep < 8; ++rep) {
          const int u = rep * 128 + tid, kk = u >> 2, c = u & 3;
          int tile, r;
          step_slot(kk, tile, r);
          const long long e = key_at(kk);
          umma::cp_async16(dst + tile * SU_A_BYTES + fp4_chunk_off(r, c),
                           a.codes + (cache_row0 + size_t(e >= 0 ? e : 0)) * 64 + 16 * c,
                           e >= 0 ? 16u : 0u);
        }
#pragma unroll
        for (int rep = 0; rep < 2; ++rep) {
          const int kk = rep * 128 + tid;
          const long long e = key_at(kk);
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;"
                       :: "r"(umma::smem_u32(Ss + s2 * SU_STEP + kk)),
                          "l"(a.scales + (cache_row0 + size_t(e >= 0 ? e : 0)) * 4),
                          "r"(e >= 0 ? 4u : 0u) : "memory");
        }
      }
      umma::cp_async_commit();
      return true;
    };
    // prefetch distance SU_STAGES - 2: the stage being refilled was read by the MMAs two
    // steps back, which have normally finished, so the producers rarely wait on them
    constexpr int PF = SU_STAGES - 2;
    bool ok = true;
    if (!a.use_tma)
      for (int g = 0; g < PF && ok; ++g) ok = issue(g);
    for (int g = 0; g < L && ok; ++g) {
      const bool new_row = g == 0 || cs.next(a);
      const int s2 = g % SU_STAGES;
      if (!a.use_tma) {   // (with the tensor map the copy thread fills the ring)
        ok = issue(g + PF);
        umma::cp_async_wait_pending(PF);    // this thread's copies for step g landed
        umma::fence_proxy_async();
        umma::mbar_arrive(&land[s2]);
      }
      if (!umma::mbar_wait(&land[s2], (g / SU_STAGES) & 1, &d_err_indexer, polls)) { ok = false; break; }
      if (new_row) {   // query scale factors: heads 0..31 in word 0 of each 4-column group
        const uint32_t qs = reinterpret_cast<const uint32_t*>(Qb + (cs.k & 1) * SU_QROW_BYTES + SU_Q_BYTES)[lane];
        const uint32_t v[8] = {sf_lo(qs), 0u, 0u, 0u, sf_hi(qs), 0u, 0u, 0u};
        umma::tmem_st8(tmem + lane_addr + SU_SFB_COL + 8 * (cs.k & 1), v);
      }
      // scale factors of rows lane, lane + 32, lane + 64, lane + 96 of both tiles; the
      // step's scale bytes are stored in step-key order
#pragma unroll
      for (int tile = 0; tile < 2; ++tile) {
        uint32_t v[8];
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
          // row 32 g4 + lane of `tile` holds step key 64 g4 + 32 tile + lane
          const uint32_t s4 = Ss[s2 * SU_STEP + 64 * g4 + 32 * tile + lane];
          v[g4] = sf_lo(s4);
          v[4 + g4] = sf_hi(s4);
        }
        umma::tmem_st8(tmem + lane_addr + SU_SFA_COL + 16 * s2 + 8 * tile, v);
      }
      umma::tmem_st_wait();
      umma::fence_before();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&sf_ready[s2]);
    }
    if (!a.use_tma) umma::cp_async_wait_all();
  } else if (warp < 8) {
    // ---------------- epilogue: warp q holds step keys 64 q .. 64 q + 63 (two tiles)
    const int q = warp & 3;
    StepCursor ce;
    ce.init(a, s_begin);
    float wv[32];
    int n_vis = 0;   // entries the current row sees (computed once per row)
    for (int g = 0; g < L; ++g) {
      const bool new_row = g == 0 || ce.next(a);
      const int row = ce.row(a);
      if (new_row) {
#pragma unroll
        for (int h = 0; h < 32; ++h) wv[h] = a.w[size_t(row) * 32 + h];
        n_vis = n_visible((long long)a.q_pos0 + ce.i, a.m, a.n_entries);
      }
      const int limit = pool ? a.row_len : n_vis;
      const int d = g % SU_ND;
      if (!umma::mbar_wait(&d_full[d], (g / SU_ND) & 1, &d_err_indexer, polls)) break;
      umma::fence_after();
      uint32_t v0[32], v1[32];
      umma::tmem_ld32(tmem + (uint32_t(q * 32) << 16) + uint32_t(64 * d), v0);
      umma::tmem_ld32(tmem + (uint32_t(q * 32) << 16) + uint32_t(64 * d + 32), v1);
      umma::tmem_ld_wait();
      umma::fence_before();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&d_empty[d]);      // accumulators copied out
      const int pbase = ce.st * SU_STEP + 64 * q + lane;
      float sc0 = 0.f, sc1 = 0.f;
#pragma unroll
      for (int h = 0; h < 32; ++h) {
        sc0 = fmaf(wv[h], fmaxf(__uint_as_float(v0[h]), 0.f), sc0);
        sc1 = fmaf(wv[h], fmaxf(__uint_as_float(v1[h]), 0.f), sc1);
      }
      float score[2] = {sc0, sc1};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int p = pbase + 32 * half;
        bool valid = p < limit;
        if (valid && pool) {
          const int cb = a.cand[size_t(row) * a.nb + p / a.blk];
          valid = cb >= 0 && cb < a.n_blocks && (long long)cb * a.blk + (p % a.blk) < n_vis;
          if (cb >= a.n_blocks) atomicOr(&d_err_indexer, ERR_BOUNDS);
        }
        if (!valid) score[half] = -INFINITY;
        if (p < a.row_len && (pool || p < n_vis)) a.scores[size_t(row) * a.row_len + p] = score[half];
      }
      if (a.blockmax) {
        // blocks of a.blk <= 64 keys lie inside one warp's 64 step keys
        if (a.blk <= 32) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float mx = score[half];
            for (int o = 1; o < a.blk; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const int p = pbase + 32 * half, bi = p / a.blk;
            if ((lane % a.blk) == 0 && bi < a.n_blocks) a.blockmax[size_t(row) * a.n_blocks + bi] = mx;
          }
        } else {
          float mx = fmaxf(score[0], score[1]);
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          const int bi = (ce.st * SU_STEP + 64 * q) / 64;
          if (lane == 0 && bi < a.n_blocks) a.blockmax[size_t(row) * a.n_blocks + bi] = mx;
        }
      }
      if (a.bm64) {   // maxima of this warp's 64 keys: a lower bound for the k-th score
        float mx = fmaxf(score[0], score[1]);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const int bi = ce.st * (SU_STEP / 64) + q;
        if (lane == 0 && bi < a.nb64) a.bm64[size_t(row) * a.nb64 + bi] = mx;
      }
    }
  } else if (warp == 8 && lane == 0) {
    // ---------------- MMA issuer: per step two tiles x two K = 64 block-scaled MMAs
    const uint32_t a0 = umma::smem_u32(As), q0 = umma::smem_u32(Qb);
    StepCursor cm;
    cm.init(a, s_begin);
    for (int g = 0; g < L; ++g) {
      // a new row: the MMAs so far are the last ones that read the other query buffer's
      // predecessor, so that buffer may be refilled once they complete
      if (g > 0 && cm.next(a)) umma::commit(&q_empty[(cm.k - 1) & 1]);
      const int s2 = g % SU_STAGES, d = g % SU_ND, qb = cm.k & 1;
      if (!umma::mbar_wait(&sf_ready[s2], (g / SU_STAGES) & 1, &d_err_indexer, polls)) break;
      if (!umma::mbar_wait(&d_empty[d], ((g / SU_ND) & 1) ^ 1, &d_err_indexer, polls)) break;
      umma::fence_after();
#pragma unroll
      for (int tile = 0; tile < 2; ++tile)
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          mma_fp4(tmem + 64 * d + 32 * tile,
                  a.use_tma ? desc_sw64(a0 + s2 * SU_STAGE_BYTES + tile * SU_A_BYTES + ks * 32)
                            : desc_noswz(a0 + s2 * SU_STAGE_BYTES + tile * SU_A_BYTES + ks * 256),
                  desc_noswz(q0 + qb * SU_QROW_BYTES + ks * 256),
                  tmem + SU_SFA_COL + 16 * s2 + 8 * tile + 4 * ks,
                  tmem + SU_SFB_COL + 8 * qb + 4 * ks, ks);
      umma::commit(&a_empty[s2]);
      umma::commit(&d_full[d]);
    }
  } else if (warp == 9 && lane == 0) {
    // ---------------- copy thread: the row's query image at each new row; with the tensor
    // map also each step as eight 2 KB tensor copies (one per 64-key block and half) plus
    // the scale bytes.  Completion is counted in bytes on land[stage]; it runs as far ahead
    // as the ring allows.
    const long long total_keys = (long long)a.rows / a.Tq * a.n_cap;   // B * n_cap
    StepCursor cc;
    cc.init(a, s_begin);
    int n_vis = 0;   // entries the current row sees (computed once per row)
    // (stall) a wait that runs out: nothing is copied, so every other role's first wait
    // runs out too and each role leaves its loop with no copy or MMA in flight
    const bool go = !a.stall || umma::mbar_wait(&never, 0, &d_err_indexer, polls);
    for (int g = 0; g < L && go; ++g) {
      const bool new_row = g == 0 || cc.next(a);
      const int s2 = g % SU_STAGES;
      if (g >= SU_STAGES &&
          !umma::mbar_wait(&a_empty[s2], ((g / SU_STAGES) - 1) & 1, &d_err_indexer, polls)) break;
      const int qb = cc.k & 1;
      if (new_row && cc.k >= 2 &&
          !umma::mbar_wait(&q_empty[qb], ((cc.k >> 1) - 1) & 1, &d_err_indexer, polls)) break;
      const int row = cc.row(a);
      if (new_row) n_vis = n_visible((long long)a.q_pos0 + cc.i, a.m, a.n_entries);
      long long blk_key[4] = {-1, -1, -1, -1};   // pool steps: the four blocks' first keys
      long long dense_key = -1;                   // dense steps: the step's first key
      uint32_t bytes = new_row ? SU_QROW_BYTES : 0u;
      if (a.use_tma) {
        const int p0 = cc.st * SU_STEP;                // first slot of the step (64-aligned)
        const int limit = pool ? a.row_len : n_vis;
        const long long cache_row0 = (long long)cc.b * a.n_cap;
        if (!pool) {
          // four consecutive blocks in two 8 KB boxes (blocks past the end of the cache
          // arrive zero-filled; keys past the visible ones are masked by the epilogue)
          if (p0 < limit) {
            dense_key = cache_row0 + p0;
            bytes += 2 * SU_A_BYTES + uint32_t(min(256ll, total_keys - dense_key)) * 4;
          }
        } else {
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            long long k0 = -1;
            if (p0 + 64 * qq < limit) {
              const int cb = a.cand[size_t(row) * a.nb + (p0 >> 6) + qq];
              if (cb >= 0 && cb < a.n_blocks) k0 = cache_row0 + 64ll * cb;
            }
            blk_key[qq] = k0;
            if (k0 >= 0) bytes += 2 * 2048 + uint32_t(min(64ll, total_keys - k0)) * 4;
          }
        }
      }
      mbar_arrive_expect_tx(&land[s2], bytes);
      if (new_row)
        bulk_load(Qb + qb * SU_QROW_BYTES, a.qprep + size_t(row) * SU_QROW_BYTES, SU_QROW_BYTES, &land[s2]);
      uint8_t* dst = As + s2 * SU_STAGE_BYTES;
      if (dense_key >= 0) {
        const int blk_id = int(dense_key >> 6);
        tma_load_4d(dst, &codes_map4, 0, 0, 0, blk_id, &land[s2]);
        tma_load_4d(dst + SU_A_BYTES, &codes_map4, 0, 0, 1, blk_id, &land[s2]);
        bulk_load(Ss + s2 * SU_STEP, a.scales + dense_key * 4,
                  uint32_t(min(256ll, total_keys - dense_key)) * 4, &land[s2]);
      }
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        if (blk_key[qq] < 0) continue;
        const int blk_id = int(blk_key[qq] >> 6);
        tma_load_4d(dst + qq * 2048, &codes_map, 0, 0, 0, blk_id, &land[s2]);
        tma_load_4d(dst + SU_A_BYTES + qq * 2048, &codes_map, 0, 0, 1, blk_id, &land[s2]);
        bulk_load(Ss + s2 * SU_STEP + 64 * qq, a.scales + blk_key[qq] * 4,
                  uint32_t(min(64ll, total_keys - blk_key[qq])) * 4, &land[s2]);
      }
    }
  }
  umma::fence_before();
  __syncthreads();
  if (warp == 0) umma::tmem_free(tmem, SU_TMEM_COLS);
}

// ---------------------------------------------------------------- prefill scoring
// Work: the (sequence, group of PF_QG queries, 128-key step) triples in order, split evenly
// over persistent CTAs (one per SM).  A step's keys (128 keys x 64 code bytes: one TMA box
// of two 64-key blocks, plus 512 scale bytes) are the MMA's A operand (M = 128); the group's
// four query images (32 heads each, consecutive in the workspace) are B (N = 128); two
// K = 64 block-scaled FP4 MMAs per step into one of three TMEM accumulators.  Sixteen
// epilogue warps (four per TMEM lane quadrant, one query each) apply ReLU and the head weights
// (packed float pairs) and store the scores of the keys each query sees.
struct GroupCursor {
  int b, g, st, n;   // sequence, group, step within the group, steps in the group
  int k;             // groups entered by this CTA so far, minus one
  __device__ void init(const ScoreArgs& a, int G, long long s) {
    const int T = a.prefix[G];
    b = int(s / T);
    const int r = int(s % T);
    int lo = 0, hi = G - 1;   // largest group with prefix <= r (that group has steps)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.prefix[mid] <= r) lo = mid; else hi = mid - 1;
    }
    g = lo;
    st = r - a.prefix[g];
    n = a.prefix[g + 1] - a.prefix[g];
    k = 0;
  }
  __device__ bool next(const ScoreArgs& a, int G) {   // only called while steps remain
    if (++st < n) return false;
    do {
      if (++g == G) { g = 0; ++b; }
      n = a.prefix[g + 1] - a.prefix[g];
    } while (n == 0);
    st = 0;
    ++k;
    return true;
  }
};

__device__ __forceinline__ float relu_dot32(const uint32_t (&v)[32], const float (&w)[32]) {
  // sum_h w_h max(s_h, 0) with packed pair FMAs into two accumulators (head pairs 4j, 4j + 1
  // and 4j + 2, 4j + 3), so that the chain of dependent FMAs is half as long
  uint64_t acc[2];
  asm("mov.b64 %0, {%1, %1};" : "=l"(acc[0]) : "f"(0.f));
  asm("mov.b64 %0, {%1, %1};" : "=l"(acc[1]) : "f"(0.f));
#pragma unroll
  for (int h = 0; h < 32; h += 2) {
    uint64_t ww, rr;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ww) : "f"(w[h]), "f"(w[h + 1]));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rr) : "f"(fmaxf(__uint_as_float(v[h]), 0.f)),
                                             "f"(fmaxf(__uint_as_float(v[h + 1]), 0.f)));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc[(h >> 1) & 1]) : "l"(ww), "l"(rr));
  }
  float x0, y0, x1, y1;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(y0) : "l"(acc[0]));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x1), "=f"(y1) : "l"(acc[1]));
  return (x0 + y0) + (x1 + y1);
}

__global__ void __launch_bounds__(PF_T, 1) score_prefill_kernel(ScoreArgs a, const uint8_t* qimg,
                                                                const uint8_t* qsc, int G,
                                                                const __grid_constant__ CUtensorMap codes_map2) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* As = base;                                                        // PF_STAGES x 8 KB
  uint32_t* Ss = reinterpret_cast<uint32_t*>(base + PF_STAGES * PF_A_BYTES); // PF_STAGES x 128 words
  uint8_t* Qb = base + PF_STAGES * (PF_A_BYTES + PF_TILE * 4);               // 2 x (image + scales)
  __shared__ __align__(8) uint64_t a_empty[PF_STAGES], land[PF_STAGES], sf_ready[PF_STAGES];
  __shared__ __align__(8) uint64_t d_full[PF_ND], d_empty[PF_ND], q_empty[2];
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long S = a.total_steps;
  const long long s_begin = S * blockIdx.x / gridDim.x, s_end = S * (blockIdx.x + 1) / gridDim.x;
  const int L = int(s_end - s_begin);
  if (L <= 0) return;   // uniform
  constexpr uint32_t QBUF = PF_Q_IMG + PF_Q_SC;

  if (tid == 0) {
    for (int s2 = 0; s2 < PF_STAGES; ++s2) {
      umma::mbar_init(&a_empty[s2], 1);
      umma::mbar_init(&land[s2], 1);
      umma::mbar_init(&sf_ready[s2], 4);
    }
    for (int d = 0; d < PF_ND; ++d) {
      umma::mbar_init(&d_full[d], 1);
      umma::mbar_init(&d_empty[d], 16);
    }
    umma::mbar_init(&q_empty[0], 1);
    umma::mbar_init(&q_empty[1], 1);
    umma::mbar_fence_init();
  }
  if (warp == 0) umma::tmem_alloc(&tmem_slot, 512);
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ---------------- copy thread: per step one TMA box of codes and the scale bytes; at a
    // new group the group's query images and scale words
    if (lane == 0) {
      const long long total_keys = (long long)(a.rows / a.Tq) * a.n_cap;   // B * n_cap
      GroupCursor cc;
      cc.init(a, G, s_begin);
      for (int g = 0; g < L; ++g) {
        const bool new_grp = g > 0 && cc.next(a, G);
        const int s2 = g % PF_STAGES;
        if (g >= PF_STAGES &&
            !umma::mbar_wait(&a_empty[s2], ((g / PF_STAGES) - 1) & 1, &d_err_indexer)) break;
        const int qb = cc.k & 1;
        if ((g == 0 || new_grp) && cc.k >= 2 &&
            !umma::mbar_wait(&q_empty[qb], ((cc.k >> 1) - 1) & 1, &d_err_indexer)) break;
        const long long key0 = (long long)cc.b * a.n_cap + (long long)cc.st * PF_TILE;
        const uint32_t sbytes = uint32_t(min((long long)PF_TILE, total_keys - key0)) * 4u;
        const bool load_q = g == 0 || new_grp;
        mbar_arrive_expect_tx(&land[s2], PF_A_BYTES + sbytes + (load_q ? QBUF : 0u));
        if (load_q) {
          const size_t r0 = size_t(cc.b) * a.Tq + size_t(cc.g) * PF_QG;   // the group's first row
          bulk_load(Qb + qb * QBUF, qimg + r0 * SU_Q_BYTES, PF_Q_IMG, &land[s2]);
          bulk_load(Qb + qb * QBUF + PF_Q_IMG, qsc + r0 * 128, PF_Q_SC, &land[s2]);
        }
        tma_load_4d(As + s2 * PF_A_BYTES, &codes_map2, 0, 0, 0, int(key0 >> 6), &land[s2]);
        bulk_load(Ss + s2 * PF_TILE, a.scales + key0 * 4, sbytes, &land[s2]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer: two K = 64 MMAs per step
    if (lane == 0) {
      const uint32_t a0 = umma::smem_u32(As), q0 = umma::smem_u32(Qb);
      GroupCursor cm;
      cm.init(a, G, s_begin);
      for (int g = 0; g < L; ++g) {
        // entering a new group: the MMAs so far are the last that read the other query
        // buffer's predecessor, which may be refilled once they complete
        if (g > 0 && cm.next(a, G)) umma::commit(&q_empty[(cm.k - 1) & 1]);
        const int s2 = g % PF_STAGES, d = g % PF_ND, qb = cm.k & 1;
        if (!umma::mbar_wait(&sf_ready[s2], (g / PF_STAGES) & 1, &d_err_indexer)) break;
        if (!umma::mbar_wait(&d_empty[d], ((g / PF_ND) & 1) ^ 1, &d_err_indexer)) break;
        umma::fence_after();
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          mma_fp4(tmem + 128 * d, desc_sw64(a0 + s2 * PF_A_BYTES + ks * 32),
                  desc_noswz(q0 + qb * QBUF + ks * 256), tmem + PF_SFA_COL + 8 * s2 + 4 * ks,
                  tmem + PF_SFB_COL + 8 * qb + 4 * ks, ks, PF_IDESC);
        umma::commit(&a_empty[s2]);
        umma::commit(&d_full[d]);
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ---------------- scale factors into TMEM (this warp's lane quadrant): the step's keys
    // (key 32 c + lane in column c of each K half) and, at a new group, its queries (head
    // lane of query c in column c)
    const uint32_t lane_addr = uint32_t((warp & 3) * 32) << 16;
    GroupCursor cs;
    cs.init(a, G, s_begin);
    for (int g = 0; g < L; ++g) {
      const bool new_grp = g > 0 && cs.next(a, G);
      const int s2 = g % PF_STAGES, qb = cs.k & 1;
      if (!umma::mbar_wait(&land[s2], (g / PF_STAGES) & 1, &d_err_indexer)) break;
      if (g == 0 || new_grp) {
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(Qb + qb * QBUF + PF_Q_IMG);
        uint32_t v[8];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t w4 = qw[32 * c + lane];
          v[c] = sf_lo(w4);
          v[4 + c] = sf_hi(w4);
        }
        umma::tmem_st8(tmem + lane_addr + PF_SFB_COL + 8 * qb, v);
      }
      uint32_t v[8];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t s4 = Ss[s2 * PF_TILE + 32 * c + lane];
        v[c] = sf_lo(s4);
        v[4 + c] = sf_hi(s4);
      }
      umma::tmem_st8(tmem + lane_addr + PF_SFA_COL + 8 * s2, v);
      umma::tmem_st_wait();
      umma::fence_before();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&sf_ready[s2]);
    }
  } else {
    // ---------------- epilogue: lane quadrant warp % 4 (keys 32 q .. 32 q + 31 of the step),
    // query qq of the group (one query per warp keeps a warp's registers to one query's
    // weights and one 32-column slice, so that sixteen warps hide each other's waits)
    const int q = warp & 3, qq = (warp - 6) >> 2;
    const uint32_t lane_addr = uint32_t(q * 32) << 16;
    GroupCursor ce;
    ce.init(a, G, s_begin);
    float w0[32];
    int nv0 = 0;   // entries this warp's query sees (0 past the last query)
    for (int g = 0; g < L; ++g) {
      const bool new_grp = g == 0 || (g > 0 && ce.next(a, G));
      const int i0 = ce.g * PF_QG + qq;                  // this warp's query index
      const size_t row0 = size_t(ce.b) * a.Tq + i0;
      const bool ok0 = i0 < a.Tq;
      if (new_grp) {
#pragma unroll
        for (int h = 0; h < 32; ++h) w0[h] = ok0 ? a.w[row0 * 32 + h] : 0.f;
        nv0 = ok0 ? n_visible((long long)a.q_pos0 + i0, a.m, a.n_entries) : 0;
      }
      const int d = g % PF_ND;
      if (!umma::mbar_wait(&d_full[d], (g / PF_ND) & 1, &d_err_indexer)) break;
      umma::fence_after();
      const int key = ce.st * PF_TILE + 32 * q + lane;
      uint32_t v[32];
      umma::tmem_ld32(tmem + lane_addr + uint32_t(128 * d + 32 * qq), v);
      umma::tmem_ld_wait();
      umma::fence_before();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&d_empty[d]);      // accumulators copied out
      const float sc0 = relu_dot32(v, w0);
      if (key < nv0) a.scores[row0 * a.row_len + key] = sc0;
    }
  }
  umma::fence_before();
  __syncthreads();
  if (warp == 0) umma::tmem_free(tmem, 512);
}

constexpr int TK_T = 512;
constexpr int TK_SMEM_KEYS = 32768;   // rows up to this length are staged in shared memory
constexpr int TK_POOL_SMEM = 1024;    // candidate blocks staged in shared memory (pool mode)

// Stage n words into shared memory with eight loads in flight per thread: the loads are
// unconditional (index clamped to n - 1) so that none waits behind a branch on another's
// value.  src[j] is converted by conv(raw) after all eight have been issued.
template <class T, class Conv, int NT = TK_T>
__device__ __forceinline__ void stage_keys(int n, unsigned* dst, const T* src, Conv conv) {
  for (int base = 0; base < n; base += 8 * NT) {
    T v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = src[min(base + u * NT + int(threadIdx.x), n - 1)];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = base + u * NT + int(threadIdx.x);
      if (j < n) dst[j] = conv(v[u]);
    }
  }
  __syncthreads();
}
__device__ __forceinline__ unsigned score_key(float f) { return (f == -INFINITY) ? 0u : f32_key(f); }

struct TopkArgs {
  const float* scores;
  int row_len, Tq, q_pos0, m, n_entries;
  const int32_t* cand;   // pool mode
  int nb, blk, k;
  int32_t* out;
};

// NT threads per row: 512 for a few long rows (latency), 256 when rows are many (more rows
// resident per SM; measured on the 16384-row prefill: 0.47 against 0.60 ms).
template <int NT>
__global__ void __launch_bounds__(NT) topk_kernel(TopkArgs a) {
  pdl_wait();
  extern __shared__ unsigned keys_sm[];
  __shared__ SelectSmem sm;
  const int row = blockIdx.x, i = row % a.Tq;
  const long long t = (long long)a.q_pos0 + i;
  const bool pool = a.cand != nullptr;
  const int n = pool ? a.row_len : n_visible(t, a.m, a.n_entries);
  const float* srow = a.scores + size_t(row) * a.row_len;
  const bool staged = n <= TK_SMEM_KEYS;
  if (staged) stage_keys<float, unsigned (*)(float), NT>(n, keys_sm, srow, score_key);
  auto key_of = [&](int j) -> unsigned { return staged ? keys_sm[j] : score_key(srow[j]); };
  int32_t* orow = a.out + size_t(row) * a.k;
  const int32_t* crow = pool ? a.cand + size_t(row) * a.nb : nullptr;
  // pool mode: the candidate blocks' first entries, in shared memory so that emitting a
  // selected slot needs no dependent global load
  __shared__ int cbase[TK_POOL_SMEM];
  const bool cstaged = pool && a.nb <= TK_POOL_SMEM;
  if (cstaged)
    for (int c = threadIdx.x; c < a.nb; c += NT) cbase[c] = crow[c] * a.blk;
  __syncthreads();
  auto emit = [&](int pos, int j) {
    int32_t v = -1;
    if (j >= 0) {
      if (!pool) v = j;
      else {
        const int c = j / a.blk;
        v = (cstaged ? cbase[c] : crow[c] * a.blk) + (j - c * a.blk);
      }
    }
    orow[pos] = v;
  };
  radix_topk<NT>(n, a.k, key_of, emit, sm);
}

// Long rows: each (row, chunk of TK_CHUNK slots) CTA selects its local top-k into a
// candidate list (keys + slot positions, in position order); a per-row merge then
// selects the top-k of the concatenated lists.  Both use the same ordering, so the
// result equals the single-pass selection.
constexpr int TK_CHUNK = 16384;

struct TopkChunkArgs {
  TopkArgs a;
  int n_chunks;
  unsigned* cand_keys;   // [rows][n_chunks][k]
  int32_t* cand_pos;     // [rows][n_chunks][k]
  const unsigned* tau;   // [rows] keys below tau cannot be among the top k (or null)
};

// Threshold from the 64-key block maxima: the k-th largest block maximum is at most the
// k-th largest score (k blocks hold a key at least that large), so keys below it can be
// dropped before selecting.  All competing keys pass when fewer than k blocks compete.
constexpr int TAU_SMEM_BLOCKS = 8192;   // rows of up to 512 Ki entries stage their maxima
__global__ void __launch_bounds__(TK_T) topk_tau_kernel(TopkArgs a, const float* bm64, int nb64,
                                                        unsigned* tau, unsigned* count) {
  pdl_wait();
  extern __shared__ unsigned bkeys[];
  __shared__ SelectSmem sm;
  const int row = blockIdx.x, i = row % a.Tq;
  const int n_vis = n_visible((long long)a.q_pos0 + i, a.m, a.n_entries);
  const int nb = (n_vis + 63) / 64;
  const float* brow = bm64 + size_t(row) * nb64;
  const bool staged = nb64 <= TAU_SMEM_BLOCKS;   // (the launch's shared memory holds nb64 keys)
  if (staged) stage_keys(nb, bkeys, brow, score_key);
  auto key_of = [&](int j) -> unsigned { return staged ? bkeys[j] : score_key(brow[j]); };
  int n_valid, k_rem;
  const unsigned kth = radix_kth<TK_T>(nb, a.k, key_of, sm, n_valid, k_rem);
  if (threadIdx.x == 0) {
    tau[row] = n_valid > a.k ? kth : 1u;
    if (count) count[row] = 0u;
  }
}

// Long dense rows, pass 1: the visible keys at or above the row's threshold, in position
// order.  CTA (row, segment of FT_SEG slots): warp w compacts its contiguous 1024 slots in
// order (ballots), then the warps' lists are concatenated into the segment's list of at most
// FT_SEGCAP entries; the segment's count is stored (a count above FT_SEGCAP marks overflow).
constexpr int FT_T = 256, FT_SEG = 8192, FT_SEGCAP = 1024, FT_WCAP = 256;
struct FilterArgs {
  TopkArgs a;
  const unsigned* tau;
  unsigned* count;      // [rows][n_seg] candidates per segment (> FT_SEGCAP: overflow)
  unsigned* ckey;       // [rows][n_seg][FT_SEGCAP]
  int32_t* cpos;        // [rows][n_seg][FT_SEGCAP]
  int n_seg;
  int stage_cap;        // candidates the final kernel's shared memory holds
};
__global__ void __launch_bounds__(FT_T) topk_filter_kernel(FilterArgs f) {
  pdl_wait();
  constexpr int NW = FT_T / 32, WSPAN = FT_SEG / NW;   // 1024 slots per warp
  __shared__ unsigned lkey[NW][FT_WCAP];
  __shared__ int32_t lpos[NW][FT_WCAP];
  __shared__ unsigned wcount[NW];
  const TopkArgs& a = f.a;
  const int row = blockIdx.x / f.n_seg, seg = blockIdx.x % f.n_seg, i = row % a.Tq;
  const int n_row = n_visible((long long)a.q_pos0 + i, a.m, a.n_entries);
  const int p0 = seg * FT_SEG;
  unsigned* cnt_out = f.count + size_t(row) * f.n_seg + seg;
  if (p0 >= n_row) {   // uniform: nothing visible in this segment
    if (threadIdx.x == 0) *cnt_out = 0u;
    return;
  }
  const unsigned thr = f.tau[row];
  const float* srow = a.scores + size_t(row) * a.row_len;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int q0 = p0 + w * WSPAN, q_end = min(q0 + WSPAN, n_row);
  unsigned n_w = 0;   // this warp's candidates so far (may exceed FT_WCAP: overflow)
  for (int base = q0; base < q_end; base += 8 * 32) {
    float v[8];   // unconditional loads (clamped index): all eight in flight at once
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = srow[max(0, min(base + u * 32 + lane, q_end - 1))];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int p = base + u * 32 + lane;
      const unsigned key = p < q_end ? score_key(v[u]) : 0u;
      const bool sel = key >= thr && key != 0u;
      const unsigned mask = __ballot_sync(0xffffffffu, sel);
      const unsigned at = n_w + unsigned(__popc(mask & ((1u << lane) - 1u)));
      if (sel && at < unsigned(FT_WCAP)) {
        lkey[w][at] = key;
        lpos[w][at] = p;
      }
      n_w += unsigned(__popc(mask));
    }
  }
  if (lane == 0) wcount[w] = n_w;
  __syncthreads();
  unsigned before = 0, total = 0;
  bool over = false;
#pragma unroll
  for (int x = 0; x < NW; ++x) {
    const unsigned c = wcount[x];
    if (x < w) before += c;
    total += c;
    over |= c > unsigned(FT_WCAP);
  }
  if (threadIdx.x == 0) *cnt_out = over ? unsigned(FT_SEGCAP) + 1u : total;
  if (over || total > unsigned(FT_SEGCAP)) return;
  unsigned* gk = f.ckey + (size_t(row) * f.n_seg + seg) * FT_SEGCAP;
  int32_t* gp = f.cpos + (size_t(row) * f.n_seg + seg) * FT_SEGCAP;
  for (unsigned j = lane; j < n_w; j += 32) {
    gk[before + j] = lkey[w][j];
    gp[before + j] = lpos[w][j];
  }
}

// Pass 2, one CTA per row: the segments' lists concatenated are in position order, so the
// radix selection's stable order (lower index first among equal keys, output ascending)
// is the method's order.  A row with an overflowing segment is selected from its full
// score row instead.
constexpr int FN_T = 256;
__global__ void __launch_bounds__(FN_T) topk_final_kernel(FilterArgs f) {
  pdl_wait();
  extern __shared__ unsigned fsm[];   // keys [n] | positions [n]
  __shared__ SelectSmem sm;
  __shared__ unsigned seg_base[129];
  __shared__ int overflow;
  __shared__ unsigned max_count;
  const TopkArgs& a = f.a;
  const int row = blockIdx.x, i = row % a.Tq, tid = threadIdx.x;
  const int n_row = n_visible((long long)a.q_pos0 + i, a.m, a.n_entries);
  const unsigned thr = f.tau[row];
  int32_t* orow = a.out + size_t(row) * a.k;
  const unsigned* cnt = f.count + size_t(row) * f.n_seg;
  if (tid < 32) {   // warp 0: the segments' offsets (lane owns segments 4 lane .. 4 lane + 3)
    unsigned c4[4], sum = 0, mx = 0;
    int ov = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = 4 * tid + u;
      c4[u] = g < f.n_seg ? cnt[g] : 0u;
      ov |= c4[u] > unsigned(FT_SEGCAP);
      if (c4[u] > unsigned(FT_SEGCAP)) c4[u] = 0u;
      sum += c4[u];
      mx = max(mx, c4[u]);
    }
    unsigned incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
      if (tid >= o) incl += y;
    }
    unsigned acc = incl - sum;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = 4 * tid + u;
      if (g < f.n_seg) seg_base[g] = acc;
      acc += c4[u];
    }
    const unsigned total = __shfl_sync(0xffffffffu, incl, 31);
    ov = __any_sync(0xffffffffu, ov);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (tid == 0) {
      seg_base[f.n_seg] = total;
      overflow = ov;
      max_count = mx;
    }
  }
  __syncthreads();
  if (overflow || seg_base[f.n_seg] > unsigned(f.stage_cap)) {   // the whole row, pruned by the threshold
    const float* srow = a.scores + size_t(row) * a.row_len;
    auto key_of = [&](int j) -> unsigned {
      const unsigned key = score_key(srow[j]);
      return key >= thr ? key : 0u;
    };
    auto emit = [&](int pos, int j) { orow[pos] = j; };
    radix_topk<FN_T>(n_row, a.k, key_of, emit, sm);
    return;
  }
  const int n = int(seg_base[f.n_seg]);
  unsigned* keys = fsm;
  int32_t* pos = reinterpret_cast<int32_t*>(fsm + f.stage_cap);
  // gather the segments in order: item x is entry x / n_seg of segment x % n_seg, so all
  // segments' loads are in flight together
  const unsigned n_items = unsigned(f.n_seg) * max_count;
  for (unsigned x = tid; x < n_items; x += FN_T) {
    const int g = int(x % unsigned(f.n_seg));
    const unsigned j = x / unsigned(f.n_seg), b0 = seg_base[g];
    if (j < seg_base[g + 1] - b0) {
      const size_t off = (size_t(row) * f.n_seg + g) * FT_SEGCAP + j;
      keys[b0 + j] = f.ckey[off];
      pos[b0 + j] = f.cpos[off];
    }
  }
  __syncthreads();
  auto key_of = [&](int j) -> unsigned { return keys[j]; };
  auto emit = [&](int slot, int j) { orow[slot] = j >= 0 ? pos[j] : -1; };
  radix_topk<FN_T>(n, a.k, key_of, emit, sm);
}

__global__ void __launch_bounds__(TK_T) topk_chunk_kernel(TopkChunkArgs c) {
  pdl_wait();
  extern __shared__ unsigned keys_sm[];
  __shared__ SelectSmem sm;
  const TopkArgs& a = c.a;
  const int row = blockIdx.x / c.n_chunks, ch = blockIdx.x % c.n_chunks, i = row % a.Tq;
  const long long t = (long long)a.q_pos0 + i;
  const int n_row = a.cand ? a.row_len : n_visible(t, a.m, a.n_entries);
  const int p0 = ch * TK_CHUNK;
  const int n = max(0, min(TK_CHUNK, n_row - p0));
  const float* srow = a.scores + size_t(row) * a.row_len + p0;
  const unsigned thr = c.tau ? c.tau[row] : 1u;
  stage_keys(n, keys_sm, srow, [&](float f) {
    const unsigned key = score_key(f);
    return key >= thr ? key : 0u;
  });
  unsigned* ck = c.cand_keys + (size_t(row) * c.n_chunks + ch) * a.k;
  int32_t* cp = c.cand_pos + (size_t(row) * c.n_chunks + ch) * a.k;
  auto key_of = [&](int j) -> unsigned { return keys_sm[j]; };
  auto emit = [&](int pos, int j) {
    ck[pos] = j >= 0 ? keys_sm[j] : 0u;
    cp[pos] = j >= 0 ? p0 + j : -1;
  };
  radix_topk<TK_T>(n, a.k, key_of, emit, sm);
}

__global__ void __launch_bounds__(TK_T) topk_merge_kernel(TopkChunkArgs c) {
  pdl_wait();
  extern __shared__ unsigned keys_sm[];
  __shared__ SelectSmem sm;
  const TopkArgs& a = c.a;
  const int row = blockIdx.x;
  const int n = c.n_chunks * a.k;
  const unsigned* ck = c.cand_keys + size_t(row) * n;
  const int32_t* cp = c.cand_pos + size_t(row) * n;
  const bool staged = n <= TK_SMEM_KEYS;
  if (staged) stage_keys(n, keys_sm, ck, [](unsigned x) { return x; });
  auto key_of = [&](int j) -> unsigned { return staged ? keys_sm[j] : ck[j]; };
  int32_t* orow = a.out + size_t(row) * a.k;
  const int32_t* crow = a.cand ? a.cand + size_t(row) * a.nb : nullptr;
  auto emit = [&](int pos, int j) {
    int32_t v = -1;
    if (j >= 0) {
      const int p = cp[j];
      v = crow ? crow[p / a.blk] * a.blk + (p % a.blk) : p;
    }
    orow[pos] = v;
  };
  radix_topk<TK_T>(n, a.k, key_of, emit, sm);
}

struct HsiArgs {
  const float* blockmax;
  int n_blocks, Tq, q_pos0, m, n_entries, blk, nb;
  int32_t* out;
};

__global__ void __launch_bounds__(TK_T) hsi_kernel(HsiArgs a) {
  pdl_wait();
  extern __shared__ unsigned bkeys[];
  __shared__ SelectSmem sm;
  const int row = blockIdx.x, i = row % a.Tq;
  const long long t = (long long)a.q_pos0 + i;
  const int n_vis = n_visible(t, a.m, a.n_entries);
  const int nb_vis = (n_vis + a.blk - 1) / a.blk;
  const int forced = n_vis > 0 ? (n_vis - 1) / a.blk : -1;
  const float* brow = a.blockmax + size_t(row) * a.n_blocks;
  const bool staged = a.n_blocks <= TAU_SMEM_BLOCKS;   // (the launch's shared memory)
  if (staged) stage_keys(nb_vis, bkeys, brow, score_key);
  auto key_of = [&](int j) -> unsigned {
    if (j == forced) return 0xFFFFFFFFu;
    return staged ? bkeys[j] : score_key(brow[j]);
  };
  int32_t* orow = a.out + size_t(row) * a.nb;
  auto emit = [&](int pos, int j) { orow[pos] = j; };
  radix_topk<TK_T>(nb_vis, a.nb, key_of, emit, sm);
}

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" {

size_t csa2_indexer_workspace_size(int B, int Tq, int n_entries, int nb, int blk, int with_cand) {
  if (B <= 0 || Tq <= 0) return 0;
  const long long row_len = with_cand ? (long long)nb * blk : n_entries;
  if (row_len <= 0) return 0;
  size_t bytes = align_up(size_t(B) * Tq * size_t(row_len) * sizeof(float), 256);
  if (row_len > TK_SMEM_KEYS) {   // candidate lists of the chunked selection, block maxima,
    const size_t n_chunks = size_t((row_len + TK_CHUNK - 1) / TK_CHUNK);   // thresholds
    bytes += 2 * align_up(size_t(B) * Tq * n_chunks * CSA2_MAX_TOPK * 4, 256);
    bytes += align_up(size_t(B) * Tq * size_t((row_len + 63) / 64) * 4, 256) +
             align_up(size_t(B) * Tq * 4, 256) +                                    // thresholds
             align_up(size_t(B) * Tq * size_t((row_len + FT_SEG - 1) / FT_SEG) * 4, 256);   // counts
  }
  // FP4 query images and the step prefix table of the tensor-core scorer
  bytes += align_up(size_t(size_t(B) * Tq + PF_QG) * SU_QROW_BYTES, 256) + align_up(size_t(Tq + 1) * 4, 256);
  return bytes;
}

int csa2_indexer_score_topk(const void* q_idx, const float* w, int B, int Tq, int q_pos0,
                            const uint8_t* codes, const uint8_t* scales, int n_cap, int n_entries,
                            int m, const int32_t* cand, int nb, int blk, int k, int32_t* topk_out,
                            float* blockmax_out, float* scores_out, void* workspace,
                            size_t ws_bytes, void* stream) {
  return csa2::indexer_impl(q_idx, w, B, Tq, q_pos0, codes, scales, n_cap, n_entries, m, cand, nb,
                            blk, k, topk_out, blockmax_out, scores_out, workspace, ws_bytes, stream,
                            nullptr, nullptr);
}

int csa2_indexer_score_topk_bounded(const void* q_idx, const float* w, int B, int Tq, int q_pos0,
                                    const uint8_t* codes, const uint8_t* scales, int n_cap,
                                    int n_entries, int m, int k, int32_t* topk_out, void* workspace,
                                    size_t ws_bytes, unsigned wait_limit, int stall, void* stream) {
  if (wait_limit == 0 && stall) return csa2::fail(CSA2_ERR_INVALID_ARG, "indexer_bounded: stall needs a wait_limit");
  // the shapes that take the tensor-core decode scorer with at least one step
  if (Tq < 1 || Tq >= csa2::PF_MIN_TQ || n_entries < 1 || m < 1 || q_pos0 + 1 < m)
    return csa2::fail(CSA2_ERR_UNSUPPORTED,
                      "indexer_bounded: needs 1 <= Tq < %d and entry 0 visible to the first query",
                      csa2::PF_MIN_TQ);
  int used = 0;
  const int st = csa2::indexer_impl(q_idx, w, B, Tq, q_pos0, codes, scales, n_cap, n_entries, m, nullptr,
                                    0, 64, k, topk_out, nullptr, nullptr, workspace, ws_bytes, stream,
                                    nullptr, nullptr, wait_limit, stall, &used);
  if (st == CSA2_OK && !used)
    return csa2::fail(CSA2_ERR_UNSUPPORTED,
                      "indexer_bounded: this call does not run the tensor-core decode scorer");
  return st;
}

}  // extern "C"

namespace {
// 4-D view of the indexer-code cache for the TMA: (64 bytes of a key) x (32 keys) x
// (2 halves) x (64-key blocks over all sequences).  A box of {64, 32, 1, nblk} lands one
// half of nblk consecutive blocks as 32 nblk rows of 64 bytes with the 64-byte swizzle:
// with nblk = 4 that is one whole MMA tile of a 256-key step.
// halves = 2: a box of whole blocks, nblk x 64 keys in key order (the prefill scorer's tiles)
bool make_codes_map(CUtensorMap* map, const uint8_t* codes, long long total_keys, int nblk, int halves = 1) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc || total_keys % 64 != 0 || total_keys / 64 > (1ll << 31) - 1) return false;
  const cuuint64_t dims[4] = {64, 32, 2, cuuint64_t(total_keys / 64)};
  const cuuint64_t strides[3] = {64, 64 * 32, 64 * 64};
  const cuuint32_t box[4] = {64, 32, cuuint32_t(halves), cuuint32_t(nblk)};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(codes), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

int csa2::indexer_impl(const void* q_idx, const float* w, int B, int Tq, int q_pos0,
                       const uint8_t* codes, const uint8_t* scales, int n_cap, int n_entries,
                       int m, const int32_t* cand, int nb, int blk, int k, int32_t* topk_out,
                       float* blockmax_out, float* scores_out, void* workspace, size_t ws_bytes,
                       void* stream, cudaEvent_t ev_score_end, cudaEvent_t ev_topk_begin,
                       unsigned wait_limit, int stall, int* used_bounded) {
  if (used_bounded) *used_bounded = 0;
  if (!q_idx || !w || !codes || !scales || !topk_out)
    return fail(CSA2_ERR_INVALID_ARG, "indexer: null tensor pointer");
  if (B <= 0 || Tq <= 0 || q_pos0 < 0 || m < 1 || n_entries < 0 || n_cap < n_entries ||
      n_cap <= 0)
    return fail(CSA2_ERR_INVALID_ARG, "indexer: bad shape B=%d Tq=%d q_pos0=%d m=%d N=%d n_cap=%d",
                B, Tq, q_pos0, m, n_entries, n_cap);
  if (k < 1 || k > CSA2_MAX_TOPK) return fail(CSA2_ERR_INVALID_ARG, "indexer: k=%d out of [1, 2048]", k);
  if (cand && blockmax_out)
    return fail(CSA2_ERR_INVALID_ARG, "indexer: blockmax is produced by Full (cand == NULL) calls only");
  if ((cand || blockmax_out) && (!is_pow2(blk) || blk > 256))
    return fail(CSA2_ERR_UNSUPPORTED, "indexer: blk=%d must be a power of two <= 256", blk);
  if (cand && (nb < 1 || nb > CSA2_MAX_TOPK))
    return fail(CSA2_ERR_INVALID_ARG, "indexer: nb=%d out of [1, 2048]", nb);
  if (!aligned16(q_idx) || !aligned16(w) || !aligned16(codes) || !aligned16(scales) ||
      !aligned16(topk_out) || (cand && !aligned16(cand)) ||
      (blockmax_out && !aligned16(blockmax_out)) || (scores_out && !aligned16(scores_out)))
    return fail(CSA2_ERR_INVALID_ARG, "indexer: pointers must be 16-byte aligned");
  const long long rows = (long long)B * Tq;
  const long long row_len = cand ? (long long)nb * blk : n_entries;
  if (rows * ((row_len + SC_CHUNK - 1) / SC_CHUNK) > (1ll << 31) - 1 || row_len > (1ll << 30) ||
      rows > (1ll << 26))
    return fail(CSA2_ERR_UNSUPPORTED, "indexer: problem too large for one call");
  // workspace: [scores unless scores_out is given][candidate lists for long rows]
  const size_t scores_bytes = align_up(size_t(rows) * size_t(row_len) * sizeof(float), 256);
  const bool chunked = row_len > TK_SMEM_KEYS;
  const size_t n_chunks_tk = chunked ? size_t((row_len + TK_CHUNK - 1) / TK_CHUNK) : 0;
  const size_t cand_bytes = chunked ? align_up(size_t(rows) * n_chunks_tk * CSA2_MAX_TOPK * 4, 256) : 0;
  // FP4 query images (+ PF_QG rows of padding: a prefill group may run past the last row)
  const size_t qprep_bytes = align_up(size_t(rows + PF_QG) * SU_QROW_BYTES, 256);
  const size_t prefix_bytes = align_up(size_t(Tq + 1) * 4, 256);
  const int nb64 = int((row_len + 63) / 64);
  const size_t bm64_bytes = chunked ? align_up(size_t(rows) * nb64 * 4, 256) : 0;
  const size_t thr_bytes = chunked ? align_up(size_t(rows) * 4, 256) : 0;
  const size_t tau_bytes = chunked ? thr_bytes + align_up(size_t(rows) * size_t((row_len + FT_SEG - 1) / FT_SEG) * 4, 256)
                                   : 0;   // thresholds + per-segment counts
  const size_t need = (scores_out ? 0 : scores_bytes) + 2 * cand_bytes + qprep_bytes + prefix_bytes +
                      bm64_bytes + tau_bytes;
  if (!workspace || ws_bytes < need || !aligned256(workspace))
    return fail(CSA2_ERR_WORKSPACE, "indexer: workspace needs %zu bytes, 256-aligned", need);
  float* scores = scores_out ? scores_out : static_cast<float*>(workspace);
  char* cand_area = static_cast<char*>(workspace) + (scores_out ? 0 : scores_bytes);
  uint8_t* qprep = reinterpret_cast<uint8_t*>(cand_area + 2 * cand_bytes);
  int* prefix = reinterpret_cast<int*>(qprep + qprep_bytes);
  float* bm64_ws = reinterpret_cast<float*>(reinterpret_cast<char*>(prefix) + prefix_bytes);
  unsigned* tau = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(bm64_ws) + bm64_bytes);
  unsigned* cand_count = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(tau) + thr_bytes);
  // long dense rows: a threshold from the 64-key block maxima prunes the chunked selection;
  // the maxima are the caller's block maxima when those are 64-key blocks
  const float* bm64_src = nullptr;
  cudaStream_t st = (cudaStream_t)stream;
  const int n_blocks = (cand || blockmax_out) ? ceil_div(n_entries, blk) : 0;
  if (row_len > 0) {
    ScoreArgs sa{(const uint16_t*)q_idx, w, int(rows), Tq, q_pos0, codes, scales, n_cap,
                 n_entries, m, cand, nb, blk, n_blocks, scores, int(row_len), blockmax_out,
                 int((row_len + SC_CHUNK - 1) / SC_CHUNK), 0, qprep, prefix, 0, nullptr, nb64,
                 umma::kWaitPolls, 0};
    const bool umma_ok = !(cand || blockmax_out) || blk <= 64;
    if (umma_ok && chunked && !cand) {
      if (blockmax_out && blk == 64) {
        bm64_src = blockmax_out;
      } else {
        sa.bm64 = bm64_ws;
        bm64_src = bm64_ws;
      }
    }
    // prefill rows (many queries per sequence, Full mode, rows short enough for the staged
    // top-k): groups of PF_QG queries share each key tile
    const bool prefill = !cand && !blockmax_out && !chunked && Tq >= PF_MIN_TQ && n_cap % 64 == 0;
    if (prefill) {
      const int G = ceil_div(Tq, PF_QG);
      long long per_seq = 0;
      for (int g = 0; g < G; ++g) {
        const int last = std::min(Tq - 1, PF_QG * g + PF_QG - 1);
        per_seq += ceil_div(n_visible((long long)q_pos0 + last, m, n_entries), PF_TILE);
      }
      sa.total_steps = per_seq * B;
      if (per_seq > (1ll << 31) - 1 || sa.total_steps > (1ll << 40))
        return fail(CSA2_ERR_UNSUPPORTED, "indexer: problem too large for one call");
      static std::atomic<int> pf_sms[64];   // SMs per device once the attribute is set
      int dev = 0;
      cudaError_t e0 = cudaGetDevice(&dev);
      if (e0 == cudaSuccess && (dev < 0 || dev >= 64)) return fail(CSA2_ERR_UNSUPPORTED, "indexer: device id");
      int sms = e0 == cudaSuccess ? pf_sms[dev].load(std::memory_order_acquire) : 0;
      if (e0 == cudaSuccess && sms == 0) {
        e0 = cudaFuncSetAttribute(score_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(PF_SMEM));
        if (e0 == cudaSuccess) e0 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e0 == cudaSuccess) pf_sms[dev].store(sms, std::memory_order_release);
      }
      if (e0 != cudaSuccess) return cuda_fail(e0, "indexer: prefill scorer attributes");
      CUtensorMap map2;
      memset(&map2, 0, sizeof(map2));
      if (!make_codes_map(&map2, codes, (long long)B * n_cap, 2, 2))
        return fail(CSA2_ERR_CUDA, "indexer: code tensor map");
      uint8_t* qimg = qprep;
      uint8_t* qsc = qprep + size_t(rows + PF_QG) * SU_Q_BYTES;
      if (sa.total_steps > 0) {
        const long long n_items = (long long)rows * 32, q_ctas = (n_items + 3) / 4;
        QPrepOut qo{qimg, SU_Q_BYTES, qsc, 128u, 1};
        CSA2_LAUNCH("q_prep launch", q_prep_kernel, unsigned(q_ctas < 4096 ? q_ctas : 4096), 128, 0, st, sa,
                    qo, prefix, n_items);
        note_launch();
        const long long grid = sa.total_steps < sms ? sa.total_steps : sms;
        CSA2_LAUNCH("score_prefill launch", score_prefill_kernel, unsigned(grid), PF_T, PF_SMEM, st, sa,
                    (const uint8_t*)qimg, (const uint8_t*)qsc, G, map2);
        note_launch();
      }
    } else if (umma_ok) {
      long long per_seq = 0;   // steps of one sequence's Tq rows (same formula as the device)
      for (int i = 0; i < Tq; ++i)
        per_seq += row_steps(i, q_pos0, m, n_entries, int(row_len), cand != nullptr, blockmax_out != nullptr);
      sa.total_steps = per_seq * B;
      if (per_seq > (1ll << 31) - 1 || sa.total_steps > (1ll << 40))
        return fail(CSA2_ERR_UNSUPPORTED, "indexer: problem too large for one call");
      static std::atomic<int> slots[64];   // resident scoring CTAs per device (0: not yet known)
      int dev = 0;
      cudaError_t e0 = cudaGetDevice(&dev);
      if (e0 == cudaSuccess && (dev < 0 || dev >= 64)) return fail(CSA2_ERR_UNSUPPORTED, "indexer: device id");
      int n_slots = e0 == cudaSuccess ? slots[dev].load(std::memory_order_acquire) : 0;
      if (e0 == cudaSuccess && n_slots == 0) {
        e0 = cudaFuncSetAttribute(score_fp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(SU_SMEM));
        if (e0 == cudaSuccess)
          e0 = cudaFuncSetAttribute(score_fp4_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        // two CTAs per SM when their shared memory fits (the launch bounds cap registers for
        // two, and their TMEM is 2 x 256 columns); the occupancy query reports one for
        // kernels that use the tensor memory, so it is not consulted
        int sms = 0, smem_sm = 0;
        if (e0 == cudaSuccess) e0 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e0 == cudaSuccess)
          e0 = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        const int per_cta = int(SU_SMEM) + 2048;   // + static shared memory and the reserved 1 KB
        if (e0 == cudaSuccess) {
          n_slots = sms * (smem_sm >= 2 * per_cta ? 2 : 1);
          slots[dev].store(n_slots, std::memory_order_release);
        }
      }
      if (e0 != cudaSuccess) return cuda_fail(e0, "indexer: scorer attributes");
      CUtensorMap map1, map4;   // boxes of one block (pool steps) and four (dense steps)
      memset(&map1, 0, sizeof(map1));
      memset(&map4, 0, sizeof(map4));
      sa.use_tma = (n_cap % 64 == 0) && (!cand || blk == 64) &&
                   make_codes_map(&map1, codes, (long long)B * n_cap, 1) &&
                   make_codes_map(&map4, codes, (long long)B * n_cap, 4);
      if (sa.total_steps > 0) {
        const long long n_items = (long long)rows * 32, q_ctas = (n_items + 3) / 4;
        QPrepOut qo{qprep, SU_QROW_BYTES, qprep + SU_Q_BYTES, SU_QROW_BYTES, 0};
        CSA2_LAUNCH("q_prep launch", q_prep_kernel, unsigned(q_ctas < 4096 ? q_ctas : 4096), 128, 0, st, sa,
                    qo, prefix, n_items);
        note_launch();
        const long long grid = sa.total_steps < n_slots ? sa.total_steps : n_slots;
        ScoreArgs sb = sa;
        if (wait_limit) sb.wait_limit = wait_limit;
        sb.stall = stall;
        CSA2_LAUNCH("score_fp4 launch", score_fp4_kernel, unsigned(grid), SU_T, SU_SMEM, st, sb, map1, map4);
        note_launch();
        if (used_bounded) *used_bounded = 1;
      }
    } else {
      CSA2_LAUNCH("score launch", score_kernel, unsigned(rows * sa.n_chunks), SC_T, 0, st, sa);
      note_launch();
    }
  }
  if (ev_score_end) record_stage_event(ev_score_end, st);
  if (ev_topk_begin) record_stage_event(ev_topk_begin, st);
  TopkArgs ta{scores, int(row_len), Tq, q_pos0, m, n_entries, cand, nb, blk, k, topk_out};
  if (!chunked) {
    const int staged = int(row_len < TK_SMEM_KEYS ? row_len : TK_SMEM_KEYS);
    const bool many = rows >= 8 * 152;   // rows to fill a 152-SM GPU eight times over
    cudaError_t e0 = cudaFuncSetAttribute(many ? topk_kernel<256> : topk_kernel<TK_T>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, TK_SMEM_KEYS * 4);
    if (e0 != cudaSuccess) return cuda_fail(e0, "indexer: top-k shared memory attribute");
    if (many) {
      CSA2_LAUNCH("topk launch", topk_kernel<256>, unsigned(rows), 256, size_t(staged) * 4, st, ta);
    } else {
      CSA2_LAUNCH("topk launch", topk_kernel<TK_T>, unsigned(rows), TK_T, size_t(staged) * 4, st, ta);
    }
    note_launch();
  } else {
    const int n_seg = int((row_len + FT_SEG - 1) / FT_SEG);
    if (bm64_src && n_seg <= 128) {
      // threshold from the block maxima, one filtering pass in position order, one exact
      // select per row (the per-segment lists fit in the chunked selection's candidate area)
      const int stage_cap = std::min(n_seg * FT_SEGCAP, 16384);
      FilterArgs fa{ta, tau, cand_count, reinterpret_cast<unsigned*>(cand_area),
                    reinterpret_cast<int32_t*>(cand_area + cand_bytes), n_seg, stage_cap};
      const size_t fsm = 2 * size_t(stage_cap) * 4;
      cudaError_t e0 = cudaFuncSetAttribute(topk_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            int(fsm));
      if (e0 != cudaSuccess) return cuda_fail(e0, "indexer: top-k shared memory attribute");
      CSA2_LAUNCH("topk_tau launch", topk_tau_kernel, unsigned(rows), TK_T, size_t(nb64 <= TAU_SMEM_BLOCKS ? nb64 : 0) * 4, st, ta, bm64_src, nb64, tau, nullptr);
      note_launch();
      CSA2_LAUNCH("topk_filter launch", topk_filter_kernel, unsigned(rows * n_seg), FT_T, 0, st, fa);
      note_launch();
      CSA2_LAUNCH("topk_final launch", topk_final_kernel, unsigned(rows), FN_T, fsm, st, fa);
      note_launch();
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_fail(e, "indexer launch");
      return CSA2_OK;
    }
    TopkChunkArgs tc{ta, int(n_chunks_tk), reinterpret_cast<unsigned*>(cand_area),
                     reinterpret_cast<int32_t*>(cand_area + cand_bytes), nullptr};
    cudaError_t e0 = cudaFuncSetAttribute(topk_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          TK_SMEM_KEYS * 4);
    if (e0 == cudaSuccess)
      e0 = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TK_SMEM_KEYS * 4);
    if (e0 != cudaSuccess) return cuda_fail(e0, "indexer: top-k shared memory attribute");
    if (rows * (long long)n_chunks_tk > (1ll << 31) - 1) return fail(CSA2_ERR_UNSUPPORTED, "indexer: too many rows");
    CSA2_LAUNCH("topk_chunk launch", topk_chunk_kernel, unsigned(rows * n_chunks_tk), TK_T, size_t(TK_CHUNK) * 4, st, tc);
    note_launch();
    const long long n_merge = (long long)n_chunks_tk * k;
    CSA2_LAUNCH("topk_merge launch", topk_merge_kernel, unsigned(rows), TK_T, size_t(n_merge <= TK_SMEM_KEYS ? n_merge : 0) * 4, st, tc);
    note_launch();
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "indexer launch");
  return CSA2_OK;
}

extern "C" {

int csa2_hsi_candidates(const float* blockmax, int B, int Tq, int q_pos0, int n_entries, int m,
                        int blk, int nb, int32_t* cand_out, void* stream) {
  if (!blockmax || !cand_out) return fail(CSA2_ERR_INVALID_ARG, "hsi: null tensor pointer");
  if (B <= 0 || Tq <= 0 || q_pos0 < 0 || m < 1 || n_entries < 0 || blk < 1)
    return fail(CSA2_ERR_INVALID_ARG, "hsi: bad shape");
  if (nb < 1 || nb > CSA2_MAX_TOPK) return fail(CSA2_ERR_INVALID_ARG, "hsi: nb=%d out of [1, 2048]", nb);
  if (!aligned16(blockmax) || !aligned16(cand_out))
    return fail(CSA2_ERR_INVALID_ARG, "hsi: pointers must be 16-byte aligned");
  const long long rows = (long long)B * Tq;
  if (rows > (1ll << 31) - 1) return fail(CSA2_ERR_UNSUPPORTED, "hsi: too many rows");
  HsiArgs ha{blockmax, ceil_div(n_entries, blk), Tq, q_pos0, m, n_entries, blk, nb, cand_out};
  CSA2_LAUNCH("hsi launch", hsi_kernel, unsigned(rows), TK_T, size_t(ha.n_blocks <= TAU_SMEM_BLOCKS ? ha.n_blocks : 0) * 4, (cudaStream_t)stream, ha);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "hsi launch");
  return CSA2_OK;
}

}  // extern "C"
