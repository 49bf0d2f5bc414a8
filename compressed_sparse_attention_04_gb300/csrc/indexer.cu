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
//   score_umma_kernel  tensor-core version of score_kernel (block <= 128): keys on M = 128,
//                  the 32 heads on N, K = 128.  Converter warps turn FP4 codes into
//                  f16 (code value times the key's block scale, exact in f16) in a
//                  128-byte-swizzled tile; one thread issues 8 tcgen05 MMAs per tile into
//                  a double-buffered TMEM accumulator; epilogue warps apply ReLU and the
//                  head weights.  All products are exact; only float32 accumulation rounds.
//   topk_kernel    one CTA per query row: radix select (select.cuh).
//   hsi_kernel     one CTA per query row: top-nb blocks with the newest block forced.
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
};

__global__ void __launch_bounds__(SC_T) score_kernel(ScoreArgs a) {
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
constexpr int SU_TILE = 128;                 // keys per tile (M)
constexpr int SU_TILES = 16;                 // tiles per CTA
constexpr int SU_STAGES = 2;                 // f16 A-tile ring
constexpr int SU_RAW = 3;                    // raw FP4 prefetch depth (tiles)
constexpr int SU_T = 288;                    // 4 converter + 4 epilogue + 1 MMA warp
constexpr uint32_t SU_A_BYTES = SU_TILE * 128 * 2;     // 32 KB
constexpr uint32_t SU_Q_BYTES = 32 * 128 * 2;          // 8 KB
constexpr uint32_t SU_RAW_STRIDE = 80;                 // bytes per key row (64 used; padded)
constexpr uint32_t SU_RAW_BYTES = SU_TILE * SU_RAW_STRIDE;   // 10 KB per stage
constexpr uint32_t SU_SMEM = SU_STAGES * SU_A_BYTES + SU_Q_BYTES + SU_RAW * SU_RAW_BYTES +
                             SU_RAW * SU_TILE * 4 + 1024;

__device__ __forceinline__ uint32_t cvt_e2m1x2_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(r) : "r"(byte));
  return r;
}
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint32_t two_bytes) {
  uint32_t r;
  asm("{\n\t.reg .b16 h;\n\tcvt.u16.u32 h, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}" : "=r"(r) : "r"(two_bytes));
  return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__global__ void __launch_bounds__(SU_T, 2) score_umma_kernel(ScoreArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* As = base;                                  // SU_STAGES x 32 KB
  uint8_t* Qs = base + SU_STAGES * SU_A_BYTES;         // 8 KB
  uint8_t* raw = Qs + SU_Q_BYTES;                      // SU_RAW x 10 KB of codes
  uint32_t* raw_sc = reinterpret_cast<uint32_t*>(raw + SU_RAW * SU_RAW_BYTES);   // SU_RAW x 128
  __shared__ __align__(8) uint64_t a_full[SU_STAGES], a_empty[SU_STAGES], d_full[2], d_empty[2];
  __shared__ __align__(8) uint64_t epi_bar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ float wmax[2][4];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = blockIdx.x / a.n_chunks, chunk = blockIdx.x % a.n_chunks;
  const int b = row / a.Tq, i = row % a.Tq;
  const long long t = (long long)a.q_pos0 + i;
  const int n_vis = n_visible(t, a.m, a.n_entries);
  const bool pool = a.cand != nullptr;
  const int limit = pool ? a.row_len : n_vis;
  const int c0 = chunk * SU_TILE * SU_TILES;
  if (c0 >= limit && a.blockmax == nullptr) return;   // uniform
  int n_tiles = SU_TILES;
  {
    const int span = (a.blockmax ? a.row_len : limit) - c0;   // slots this CTA must cover
    const int need = span <= 0 ? 1 : (span + SU_TILE - 1) / SU_TILE;
    n_tiles = need < SU_TILES ? need : SU_TILES;
  }

  // query -> FP4 (same rule as the keys) -> f16 B operand (32 heads x 128, K-major)
  const uint16_t* qrow = a.q_idx + size_t(row) * 32 * 128;
  for (int pb = warp; pb < 128; pb += SU_T / 32) {
    const int h = pb >> 2, blk4 = pb & 3;
    const float v = bf16_to_f32(qrow[h * 128 + blk4 * 32 + lane]);
    uint32_t sb;
    const uint32_t code = fp4_quant_lane(v, sb);
    const __half qv = __float2half_rn(e2m1_value(code) * e4m3_value(sb));   // exact
    *reinterpret_cast<__half*>(Qs + umma::kmajor_sw128_offset(h, blk4 * 32 + lane, 32)) = qv;
  }
  if (tid == 0) {
    for (int s2 = 0; s2 < SU_STAGES; ++s2) { umma::mbar_init(&a_full[s2], 4); umma::mbar_init(&a_empty[s2], 1); }
    for (int d = 0; d < 2; ++d) {
      umma::mbar_init(&d_full[d], 1);
      umma::mbar_init(&d_empty[d], 4);
      umma::mbar_init(&epi_bar[d], 4);
    }
    umma::mbar_fence_init();
  }
  if (warp == 0) umma::tmem_alloc(&tmem_slot, 64);
  umma::fence_proxy_async();
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
  const uint32_t tmem = tmem_slot;
  const size_t cache_row0 = size_t(b) * a.n_cap;

  if (warp < 4) {
    // ---------------- converters: thread = key of the tile.  Each thread prefetches
    // its own key's 64 code bytes and 4 scale bytes SU_RAW - 1 tiles ahead with
    // asynchronous copies, then writes the f16 row into the swizzled A tile.
    auto key_of = [&](int j) -> long long {
      const int p = c0 + j * SU_TILE + tid;
      if (j >= n_tiles || p >= limit) return -1;
      if (!pool) return p;
      const int cb = a.cand[size_t(row) * a.nb + p / a.blk];
      if (cb < 0 || cb >= a.n_blocks) return -1;
      const long long ee = (long long)cb * a.blk + (p % a.blk);
      return ee < n_vis ? ee : -1;
    };
    auto issue = [&](int j) {
      const long long e = key_of(j);
      if (e >= 0) {
        const uint8_t* src = a.codes + (cache_row0 + size_t(e)) * 64;
        uint8_t* dst = raw + (j % SU_RAW) * SU_RAW_BYTES + tid * SU_RAW_STRIDE;
#pragma unroll
        for (int u = 0; u < 4; ++u) umma::cp_async16(dst + 16 * u, src + 16 * u, 16u);
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;"
                     :: "r"(umma::smem_u32(raw_sc + (j % SU_RAW) * SU_TILE + tid)),
                        "l"(a.scales + (cache_row0 + size_t(e)) * 4) : "memory");
      }
      umma::cp_async_commit();
    };
    for (int j = 0; j < SU_RAW - 1; ++j) issue(j);
    for (int j = 0; j < n_tiles; ++j) {
      issue(j + SU_RAW - 1);
      umma::cp_async_wait_pending(SU_RAW - 1);   // this thread's tile-j copies landed
      const int s2 = j % SU_STAGES;
      if (!umma::mbar_wait(&a_empty[s2], ((j / SU_STAGES) & 1) ^ 1, &d_err_indexer)) break;
      uint8_t* arow = As + s2 * SU_A_BYTES;
      if (key_of(j) >= 0) {
        const uint8_t* rsrc = raw + (j % SU_RAW) * SU_RAW_BYTES + tid * SU_RAW_STRIDE;
        const uint32_t sc4 = raw_sc[(j % SU_RAW) * SU_TILE + tid];
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          const uint4 cvv = *reinterpret_cast<const uint4*>(rsrc + 16 * kb);
          const uint32_t sbyte = (sc4 >> (8 * kb)) & 0xFFu;
          const uint32_t s2h = cvt_e4m3x2_f16x2(sbyte | (sbyte << 8));
          const uint32_t w4[4] = {cvv.x, cvv.y, cvv.z, cvv.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {      // 8 codes -> 8 f16 -> one 16-byte chunk
            uint32_t o[4];
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) o[bb] = hmul2(cvt_e2m1x2_f16x2((w4[u] >> (8 * bb)) & 0xFFu), s2h);
            const int k = kb * 32 + u * 8;
            *reinterpret_cast<uint4*>(arow + umma::kmajor_sw128_offset(tid, k, SU_TILE)) =
                make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
      umma::fence_proxy_async();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&a_full[s2]);
    }
    umma::cp_async_wait_all();
  } else if (warp < 8) {
    // ---------------- epilogue: thread = key of the tile (lane quadrant warp % 4)
    const int q = warp & 3;
    float wv[32];
#pragma unroll
    for (int h = 0; h < 32; ++h) wv[h] = a.w[size_t(row) * 32 + h];
    for (int j = 0; j < n_tiles; ++j) {
      const int d = j & 1;
      if (!umma::mbar_wait(&d_full[d], (j >> 1) & 1, &d_err_indexer)) break;
      umma::fence_after();
      uint32_t v[32];
      umma::tmem_ld32(tmem + (uint32_t(q * 32) << 16) + uint32_t(32 * d), v);
      umma::tmem_ld_wait();
      umma::fence_before();
      const int p = c0 + j * SU_TILE + q * 32 + lane;
      bool valid = p < limit;
      if (valid && pool) {
        const int cb = a.cand[size_t(row) * a.nb + p / a.blk];
        valid = cb >= 0 && cb < a.n_blocks && (long long)cb * a.blk + (p % a.blk) < n_vis;
        if (cb >= a.n_blocks) atomicOr(&d_err_indexer, ERR_BOUNDS);
      }
      float sc = 0.f;
#pragma unroll
      for (int h = 0; h < 32; ++h) sc = fmaf(wv[h], fmaxf(__uint_as_float(v[h]), 0.f), sc);
      const float score = valid ? sc : -INFINITY;
      if (p < a.row_len && (pool || p < n_vis)) a.scores[size_t(row) * a.row_len + p] = score;
      if (a.blockmax) {
        // blocks of a.blk keys (power of two <= 128) never straddle a 128-key tile
        float mx = score;
        const int gl = a.blk < 32 ? a.blk : 32;
        for (int o = 1; o < gl; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (a.blk <= 32) {
          const int bi = p / a.blk;
          if ((lane % a.blk) == 0 && bi < a.n_blocks) a.blockmax[size_t(row) * a.n_blocks + bi] = mx;
        } else {
          if (lane == 0) wmax[d][q] = mx;
          __syncwarp();
          if (lane == 0) umma::mbar_arrive(&epi_bar[d]);
          if (!umma::mbar_wait(&epi_bar[d], (j >> 1) & 1, &d_err_indexer)) break;
          if (lane == 0 && (q % (a.blk / 32)) == 0) {
            float m2 = mx;
            for (int u = 1; u < a.blk / 32; ++u) m2 = fmaxf(m2, wmax[d][q + u]);
            const int bi = p / a.blk;
            if (bi < a.n_blocks) a.blockmax[size_t(row) * a.n_blocks + bi] = m2;
          }
        }
      }
      // the TMEM buffer and wmax[d] are reused two tiles later: release both now
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&d_empty[d]);
    }
  } else if (lane == 0) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc = umma::idesc_f16(SU_TILE, 32, 0, 0, 0);
    const uint32_t a0 = umma::smem_u32(As), q0 = umma::smem_u32(Qs);
    for (int j = 0; j < n_tiles; ++j) {
      const int s2 = j % SU_STAGES, d = j & 1;
      if (!umma::mbar_wait(&a_full[s2], (j / SU_STAGES) & 1, &d_err_indexer)) break;
      if (!umma::mbar_wait(&d_empty[d], ((j >> 1) & 1) ^ 1, &d_err_indexer)) break;
      umma::fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t da = umma::desc_sw128(a0 + s2 * SU_A_BYTES + (kk >> 2) * (SU_TILE * 128) + (kk & 3) * 32, 16, 1024);
        const uint64_t db = umma::desc_sw128(q0 + (kk >> 2) * (32 * 128) + (kk & 3) * 32, 16, 1024);
        umma::mma_f16(tmem + 32 * d, da, db, idesc, kk > 0);
      }
      umma::commit(&a_empty[s2]);
      umma::commit(&d_full[d]);
    }
  }
  umma::fence_before();
  __syncthreads();
  if (warp == 0) umma::tmem_free(tmem, 64);
}

constexpr int TK_T = 512;
constexpr int TK_SMEM_KEYS = 32768;   // rows up to this length are staged in shared memory

struct TopkArgs {
  const float* scores;
  int row_len, Tq, q_pos0, m, n_entries;
  const int32_t* cand;   // pool mode
  int nb, blk, k;
  int32_t* out;
};

__global__ void __launch_bounds__(TK_T) topk_kernel(TopkArgs a) {
  extern __shared__ unsigned keys_sm[];
  __shared__ SelectSmem sm;
  const int row = blockIdx.x, i = row % a.Tq;
  const long long t = (long long)a.q_pos0 + i;
  const bool pool = a.cand != nullptr;
  const int n = pool ? a.row_len : n_visible(t, a.m, a.n_entries);
  const float* srow = a.scores + size_t(row) * a.row_len;
  const bool staged = n <= TK_SMEM_KEYS;
  if (staged) {
    for (int j = threadIdx.x; j < n; j += TK_T) {
      const float f = srow[j];
      keys_sm[j] = (f == -INFINITY) ? 0u : f32_key(f);
    }
    __syncthreads();
  }
  auto key_of = [&](int j) -> unsigned {
    if (staged) return keys_sm[j];
    const float f = srow[j];
    return (f == -INFINITY) ? 0u : f32_key(f);
  };
  int32_t* orow = a.out + size_t(row) * a.k;
  const int32_t* crow = pool ? a.cand + size_t(row) * a.nb : nullptr;
  auto emit = [&](int pos, int j) {
    int32_t v = -1;
    if (j >= 0) v = pool ? crow[j / a.blk] * a.blk + (j % a.blk) : j;
    orow[pos] = v;
  };
  radix_topk<TK_T>(n, a.k, key_of, emit, sm);
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
};

__global__ void __launch_bounds__(TK_T) topk_chunk_kernel(TopkChunkArgs c) {
  extern __shared__ unsigned keys_sm[];
  __shared__ SelectSmem sm;
  const TopkArgs& a = c.a;
  const int row = blockIdx.x / c.n_chunks, ch = blockIdx.x % c.n_chunks, i = row % a.Tq;
  const long long t = (long long)a.q_pos0 + i;
  const int n_row = a.cand ? a.row_len : n_visible(t, a.m, a.n_entries);
  const int p0 = ch * TK_CHUNK;
  const int n = max(0, min(TK_CHUNK, n_row - p0));
  const float* srow = a.scores + size_t(row) * a.row_len + p0;
  for (int j = threadIdx.x; j < n; j += TK_T) {
    const float f = srow[j];
    keys_sm[j] = (f == -INFINITY) ? 0u : f32_key(f);
  }
  __syncthreads();
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
  extern __shared__ unsigned keys_sm[];
  __shared__ SelectSmem sm;
  const TopkArgs& a = c.a;
  const int row = blockIdx.x;
  const int n = c.n_chunks * a.k;
  const unsigned* ck = c.cand_keys + size_t(row) * n;
  const int32_t* cp = c.cand_pos + size_t(row) * n;
  const bool staged = n <= TK_SMEM_KEYS;
  if (staged) {
    for (int j = threadIdx.x; j < n; j += TK_T) keys_sm[j] = ck[j];
    __syncthreads();
  }
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
  __shared__ SelectSmem sm;
  const int row = blockIdx.x, i = row % a.Tq;
  const long long t = (long long)a.q_pos0 + i;
  const int n_vis = n_visible(t, a.m, a.n_entries);
  const int nb_vis = (n_vis + a.blk - 1) / a.blk;
  const int forced = n_vis > 0 ? (n_vis - 1) / a.blk : -1;
  const float* brow = a.blockmax + size_t(row) * a.n_blocks;
  auto key_of = [&](int j) -> unsigned {
    if (j == forced) return 0xFFFFFFFFu;
    const float f = brow[j];
    return (f == -INFINITY) ? 0u : f32_key(f);
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
  if (row_len > TK_SMEM_KEYS) {   // candidate lists of the chunked selection
    const size_t n_chunks = size_t((row_len + TK_CHUNK - 1) / TK_CHUNK);
    bytes += 2 * align_up(size_t(B) * Tq * n_chunks * CSA2_MAX_TOPK * 4, 256);
  }
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

}  // extern "C"

int csa2::indexer_impl(const void* q_idx, const float* w, int B, int Tq, int q_pos0,
                       const uint8_t* codes, const uint8_t* scales, int n_cap, int n_entries,
                       int m, const int32_t* cand, int nb, int blk, int k, int32_t* topk_out,
                       float* blockmax_out, float* scores_out, void* workspace, size_t ws_bytes,
                       void* stream, cudaEvent_t ev_score_end, cudaEvent_t ev_topk_begin) {
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
  if (rows * ((row_len + SC_CHUNK - 1) / SC_CHUNK) > (1ll << 31) - 1 || row_len > (1ll << 30))
    return fail(CSA2_ERR_UNSUPPORTED, "indexer: problem too large for one call");
  // workspace: [scores unless scores_out is given][candidate lists for long rows]
  const size_t scores_bytes = align_up(size_t(rows) * size_t(row_len) * sizeof(float), 256);
  const bool chunked = row_len > TK_SMEM_KEYS;
  const size_t n_chunks_tk = chunked ? size_t((row_len + TK_CHUNK - 1) / TK_CHUNK) : 0;
  const size_t cand_bytes = chunked ? align_up(size_t(rows) * n_chunks_tk * CSA2_MAX_TOPK * 4, 256) : 0;
  const size_t need = (scores_out ? 0 : scores_bytes) + 2 * cand_bytes;
  if (need && (!workspace || ws_bytes < need || !aligned256(workspace)))
    return fail(CSA2_ERR_WORKSPACE, "indexer: workspace needs %zu bytes, 256-aligned", need);
  float* scores = scores_out ? scores_out : static_cast<float*>(workspace);
  char* cand_area = static_cast<char*>(workspace) + (scores_out ? 0 : scores_bytes);
  cudaStream_t st = (cudaStream_t)stream;
  const int n_blocks = (cand || blockmax_out) ? ceil_div(n_entries, blk) : 0;
  if (row_len > 0) {
    ScoreArgs sa{(const uint16_t*)q_idx, w, int(rows), Tq, q_pos0, codes, scales, n_cap,
                 n_entries, m, cand, nb, blk, n_blocks, scores, int(row_len), blockmax_out,
                 int((row_len + SC_CHUNK - 1) / SC_CHUNK)};
    const bool umma_ok = !(cand || blockmax_out) || blk <= 128;
    if (umma_ok) {
      sa.n_chunks = int((row_len + SU_TILE * SU_TILES - 1) / (SU_TILE * SU_TILES));
      cudaError_t e0 = cudaFuncSetAttribute(score_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            int(SU_SMEM));
      if (e0 != cudaSuccess) return cuda_fail(e0, "indexer: shared memory attribute");
      score_umma_kernel<<<unsigned(rows * sa.n_chunks), SU_T, SU_SMEM, st>>>(sa);
    } else {
      score_kernel<<<unsigned(rows * sa.n_chunks), SC_T, 0, st>>>(sa);
    }
  }
  if (ev_score_end) cudaEventRecord(ev_score_end, st);
  if (ev_topk_begin) cudaEventRecord(ev_topk_begin, st);
  TopkArgs ta{scores, int(row_len), Tq, q_pos0, m, n_entries, cand, nb, blk, k, topk_out};
  if (!chunked) {
    const int staged = int(row_len < TK_SMEM_KEYS ? row_len : TK_SMEM_KEYS);
    cudaError_t e0 = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          TK_SMEM_KEYS * 4);
    if (e0 != cudaSuccess) return cuda_fail(e0, "indexer: top-k shared memory attribute");
    topk_kernel<<<unsigned(rows), TK_T, size_t(staged) * 4, st>>>(ta);
  } else {
    TopkChunkArgs tc{ta, int(n_chunks_tk), reinterpret_cast<unsigned*>(cand_area),
                     reinterpret_cast<int32_t*>(cand_area + cand_bytes)};
    cudaError_t e0 = cudaFuncSetAttribute(topk_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          TK_SMEM_KEYS * 4);
    if (e0 == cudaSuccess)
      e0 = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TK_SMEM_KEYS * 4);
    if (e0 != cudaSuccess) return cuda_fail(e0, "indexer: top-k shared memory attribute");
    if (rows * (long long)n_chunks_tk > (1ll << 31) - 1) return fail(CSA2_ERR_UNSUPPORTED, "indexer: too many rows");
    topk_chunk_kernel<<<unsigned(rows * n_chunks_tk), TK_T, size_t(TK_CHUNK) * 4, st>>>(tc);
    const long long n_merge = (long long)n_chunks_tk * k;
    topk_merge_kernel<<<unsigned(rows), TK_T, size_t(n_merge <= TK_SMEM_KEYS ? n_merge : 0) * 4, st>>>(tc);
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
  hsi_kernel<<<unsigned(rows), TK_T, 0, (cudaStream_t)stream>>>(ha);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "hsi launch");
  return CSA2_OK;
}

}  // extern "C"
