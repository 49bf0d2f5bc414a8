// Stage 1 (compressor) and stage 2 (indexer key + FP4) of the CSA2 hot path.
//
// [P1] "DeepSeek-V4.1 模型结构（2）：序列维度（中），CSA2 的三种模式" (blog.javazero.top):
//      §压缩算子去掉了重叠和位置偏置 -- disjoint groups of m tokens, per-channel softmax
//      pooling, no position bias, m = 1 without a gate, RMSNorm, RoPE on the last 64
//      dims at the group's first token; §indexer K 改由 main KV 投影 -- indexer key
//      projected 512 -> 128 from the entry before RoPE, its own RoPE on the last 64
//      dims, no Hadamard, FP4 with one scale per 32 dims.
// [P2] "DeepSeek v4.1 Flash技术剖析——架构篇" (myhz0606.com) §Compressor.
//
// Kernels
//   proj_umma_kernel   P[split][M, Nout] = X[M, K-range] . [W_kv; W_gate]^T on tcgen05: one CTA
//                      per (128 channels, 128 rows, K-range); D^T = W X^T in TMEM; a 4-stage
//                      cp.async pipeline feeds 128B-swizzled tiles; the K-ranges (split-K,
//                      used when there are few rows, as in decode) are summed in fixed order
//                      by the epilogue, so results do not depend on scheduling.
//   proj_gemm_kernel   SIMT fallback of the same product
//   compress_epilogue  per entry: softmax-pool over the group, RMSNorm, RoPE, stores; with a
//                      group state (csa2_compress_chunk) also the entry a previous call's
//                      token started and the stash of a group this call leaves open
//   index_k_kernel     per entry: 512 -> 128 projection, RoPE, FP4 quantisation
//   main_kv_fp4_kernel per entry: the stored main-KV entry as FP4 (E2M1 codes, one E4M3
//                      scale per 16 channels: 288 bytes)
//   swa_kv_fp8_kernel  per window row: FP8 (E4M3 codes, one power-of-two scale per 64
//                      channels: 520 bytes)
#include "common.cuh"
#include "umma.cuh"

CSA2_DEFINE_ERR_WORD(d_err_compress)

namespace csa2 {
namespace {

constexpr int GM = 128, GN = 128, GK = 32, GT = 256;

// Register-tiled SIMT GEMM.  Each of 256 threads owns an 8x8 sub-tile with rows
// ty + 16 i and columns tx + 16 j; tiles staged in shared memory as float32, K-major.
__global__ void __launch_bounds__(GT) proj_gemm_kernel(const uint16_t* __restrict__ X,
                                                       const uint16_t* __restrict__ W0,
                                                       const uint16_t* __restrict__ W1, int M,
                                                       int K, int Nout, float* __restrict__ P) {
  pdl_wait();
  __shared__ float As[GK][GM + 4];
  __shared__ float Bs[GK][GN + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * GM, n0 = blockIdx.x * GN;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += GK) {
    // 128 rows x 32 k = 512 chunks of 8 bf16; 2 chunks per thread for A and for B
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int chunk = tid + c * GT, r = chunk >> 2, kc = (chunk & 3) * 8;
      uint4 va = make_uint4(0, 0, 0, 0);
      if (m0 + r < M) va = *reinterpret_cast<const uint4*>(X + size_t(m0 + r) * K + k0 + kc);
      const int n = n0 + r;
      const uint16_t* wrow = (n < 512) ? (W0 + size_t(n) * K) : (W1 + size_t(n - 512) * K);
      uint4 vb = *reinterpret_cast<const uint4*>(wrow + k0 + kc);
      const uint16_t* pa = reinterpret_cast<const uint16_t*>(&va);
      const uint16_t* pb = reinterpret_cast<const uint16_t*>(&vb);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        As[kc + u][r] = bf16_to_f32(pa[u]);
        Bs[kc + u][r] = bf16_to_f32(pb[u]);
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < GK; ++kk) {
      float a[8], b[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 8; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = m0 + ty + 16 * i;
    if (r >= M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) P[size_t(r) * Nout + n0 + tx + 16 * j] = acc[i][j];
  }
}


constexpr int PU_T = 128;
constexpr int PU_TILE = 128;                 // channels (M of the MMA) and rows (N)
constexpr int PU_KC = 64;                    // K per stage (one 128-byte atom column)
constexpr int PU_STAGES = 4;
constexpr uint32_t PU_STAGE_BYTES = 2 * PU_TILE * PU_KC * 2;   // 32 KB (W tile + X tile)
constexpr uint32_t PU_SMEM = PU_STAGES * PU_STAGE_BYTES + 1024;

// Operand tiles by TMA (128-byte swizzle, the layout the MMA descriptors read): thread 0 of
// warp 0 keeps PU_STAGES stages of (W tile, X tile) in flight on full / empty mbarriers,
// thread 0 of warp 1 issues the MMAs; X rows past M arrive as zeros.  W rows n < 512 come
// from w_kv, the others from w_gate (a 128-channel tile lies in one of them).
__device__ __forceinline__ void pu_tma_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];"
      :: "r"(umma::smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(umma::smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void pu_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
               :: "r"(umma::smem_u32(bar)), "r"(bytes) : "memory");
}

__global__ void __launch_bounds__(PU_T, 1) proj_umma_kernel(const __grid_constant__ CUtensorMap x_map,
                                                            const __grid_constant__ CUtensorMap w0_map,
                                                            const __grid_constant__ CUtensorMap w1_map,
                                                            int M, int Nout, int k_per_split,
                                                            float* __restrict__ P) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[PU_STAGES], empty_bar[PU_STAGES], done_bar;
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * PU_TILE;            // channel tile
  const int m0 = blockIdx.y * PU_TILE;            // row tile
  const int split = blockIdx.z;
  const int k_begin = split * k_per_split;
  const int n_iter = k_per_split / PU_KC;
  if (tid == 0) {
    for (int s = 0; s < PU_STAGES; ++s) {
      umma::mbar_init(&full_bar[s], 1);
      umma::mbar_init(&empty_bar[s], 1);
    }
    umma::mbar_init(&done_bar, 1);
    umma::mbar_fence_init();
  }
  if (warp == 0) umma::tmem_alloc(&tmem_slot, 128);
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;
  int issued = 0;                                  // producer: stages loaded so far
  if (warp == 0 && lane == 0) {
    // ---------------- producer
    const CUtensorMap* wmap = n0 < 512 ? &w0_map : &w1_map;
    const int wy = n0 < 512 ? n0 : n0 - 512;
    for (int it = 0; it < n_iter; ++it, ++issued) {
      const int s = it % PU_STAGES;
      if (it >= PU_STAGES &&
          !umma::mbar_wait(&empty_bar[s], ((it / PU_STAGES) - 1) & 1, &d_err_compress)) { ok = false; break; }
      uint8_t* Ws = base + s * PU_STAGE_BYTES;
      uint8_t* Xs = Ws + PU_TILE * PU_KC * 2;
      const int k0 = k_begin + it * PU_KC;
      pu_expect_tx(&full_bar[s], PU_STAGE_BYTES);
      pu_tma_2d(Ws, wmap, k0, wy, &full_bar[s]);
      pu_tma_2d(Xs, &x_map, k0, m0, &full_bar[s]);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc = umma::idesc_f16(PU_TILE, PU_TILE, 1, 0, 0);
    for (int it = 0; it < n_iter; ++it) {
      const int s = it % PU_STAGES;
      if (!umma::mbar_wait(&full_bar[s], (it / PU_STAGES) & 1, &d_err_compress)) { ok = false; break; }
      umma::fence_after();
      const uint32_t wb = umma::smem_u32(base + s * PU_STAGE_BYTES);
      const uint32_t xb = wb + PU_TILE * PU_KC * 2;
#pragma unroll
      for (int kk = 0; kk < PU_KC / 16; ++kk)
        umma::mma_f16(tmem, umma::desc_sw128(wb + kk * 32, 16, 1024),
                      umma::desc_sw128(xb + kk * 32, 16, 1024), idesc, (it | kk) != 0);
      umma::commit(&empty_bar[s]);
    }
    umma::commit(&done_bar);   // (all MMAs issued by this thread, also after an early stop)
  }
  __syncwarp();
  ok = umma::mbar_wait(&done_bar, 0, &d_err_compress) && ok;
  ok = __syncthreads_and(ok);
  if (!ok && warp == 0 && lane == 0) {
    // a wait gave up: let the copies still in flight land before the CTA leaves
    for (int it = issued - 1; it >= 0 && it >= issued - PU_STAGES; --it)
      umma::mbar_wait(&full_bar[it % PU_STAGES], (it / PU_STAGES) & 1, &d_err_compress);
  }
  umma::fence_after();
  if (ok) {
    // D^T: lane = channel n0 + 32*warp + lane, column = row m0 + c
    const int n = n0 + warp * 32 + lane;
    float* Pd = P + size_t(split) * size_t(M) * Nout;
#pragma unroll 1
    for (int c0 = 0; c0 < PU_TILE; c0 += 32) {
      uint32_t v[32];
      umma::tmem_ld32(tmem + (uint32_t(warp * 32) << 16) + uint32_t(c0), v);
      umma::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int m = m0 + c0 + c;
        if (m < M) Pd[size_t(m) * Nout + n] = __uint_as_float(v[c]);
      }
    }
  }
  umma::fence_before();
  __syncthreads();
  if (warp == 0) umma::tmem_free(tmem, 128);
}

int proj_splits(int M, int K, int Nout) {
  const int tiles = (Nout / PU_TILE) * ((M + PU_TILE - 1) / PU_TILE);
  int s = 1;
  while (s * 2 <= K / 256 && tiles * s * 2 <= 2 * 152 && (K / PU_KC) % (s * 2) == 0) s *= 2;
  return s;
}

// Quarter qk of key dim j of one entry: sum over inputs 128 qk .. 128 qk + 127 of
// w_ik[j][i] * y[i], in input order; quarters 1..3 go to ipart (after a barrier that the
// caller's quarter 0 meets), quarter 0 is returned once they are there.
__device__ __forceinline__ float idx_quarter(const float* ys, const uint4* wv, int qk, int j,
                                             float (*ipart)[128]) {
  float acc = 0.f;
#pragma unroll
  for (int u8 = 0; u8 < 16; ++u8) {
    const uint16_t* pv = reinterpret_cast<const uint16_t*>(&wv[u8]);
#pragma unroll
    for (int u = 0; u < 8; ++u) acc = fmaf(bf16_to_f32(pv[u]), ys[128 * qk + 8 * u8 + u], acc);
  }
  if (qk > 0) ipart[qk - 1][j] = acc;
  __syncthreads();
  return acc;
}
// Key dim j (thread j of the first 128) of entry `ent`: RoPE on dims 64..127 at position
// ent * m, FP4 codes (two per byte) and the E4M3 scale of each 32-dim block.
__device__ __forceinline__ void idx_finish(float v, int j, long long ent, int m, const RopeTurns& rt,
                                           uint8_t* codes, uint8_t* scales, size_t crow,
                                           float* k_out, size_t k_row) {
  const int lane = j & 31, w = j >> 5;
  const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
  if (j >= 64) {
    float c, s;
    rope_cs(ent * m, (j - 64) >> 1, rt, c, s);
    v = (j & 1) ? (partner * s + v * c) : (v * c - partner * s);
  }
  if (k_out) k_out[k_row * 128 + j] = v;
  uint32_t sb;
  const uint32_t code = fp4_quant_lane(v, sb);
  const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
  if ((lane & 1) == 0) codes[crow * 64 + (j >> 1)] = uint8_t(code | (hi << 4));
  if (lane == 0) scales[crow * 4 + w] = uint8_t(sb);
}

// One block of 512 threads per entry: thread t < 128 of split group sg = tid / 128 sums
// channels 4t..4t+3 of splits [sg * n / 4, (sg + 1) * n / 4) of the n_split partial products
// (split-K), all its loads in flight together; group 0 then adds the four group sums in group
// order and finishes the entry (the summation order is fixed: deterministic).
// A chunk holds tokens pos0 .. pos0+T-1 of each sequence (rows b*T .. b*T+T-1 of P).  Per
// sequence, block r < n_ent writes entry pos0/m + r; with head = 1 (m = 2, pos0 odd) block 0
// completes the group whose first token the previous chunk left in `state`.  With tail = 1 (the
// chunk ends inside a group) the last token's kv and gate sums go to state: from block 0 when
// head = 1 (which reads the old state first: one block per sequence touches it), else from an
// extra block r = n_ent.
// With IDX (few entries, as in decode) the block also computes the entry's indexer key from
// the pre-RoPE entry it holds, exactly as index_k_kernel does (same products, same order):
// the 512 threads split the 512 -> 128 projection into four quarters of the inputs, the
// first 128 add them in quarter order, apply RoPE and quantise to FP4.
struct IdxOut {
  const uint16_t* w_ik;   // [128][512] bf16
  uint8_t* codes;         // [B][n_cap][64]
  uint8_t* scales;        // [B][n_cap][4]
};
template <bool IDX>
__global__ void __launch_bounds__(512) compress_epilogue_kernel(
    const float* __restrict__ P, int n_split, size_t split_stride, int Nout, int T, int m,
    int pos0, int n_ent, int head, int tail,
    const float* __restrict__ norm_w, float eps, const RopeTurns rt, uint16_t* __restrict__ kv_cache,
    int n_cap, float* __restrict__ kv_pre, float* __restrict__ state, IdxOut io) {
  pdl_wait();
  __shared__ float4 part[3][128][4];   // groups 1..3: their sums per thread
  __shared__ float ys[IDX ? 512 : 1];           // (IDX) the entry before RoPE
  __shared__ float ipart[IDX ? 3 : 1][128];     // (IDX) quarter sums of the key projection
  const int per = n_ent + (tail && !head ? 1 : 0);
  const int b = blockIdx.x / per, r = blockIdx.x % per, t = threadIdx.x & 127, sg = threadIdx.x >> 7;
  const bool from_state = head && r == 0, to_state = r == n_ent, stash_too = from_state && tail;
  // (IDX) this thread's 128 key-projection weights: row t, inputs 128 sg .. 128 sg + 127, in
  // flight while the entry is computed
  uint4 wv[IDX ? 16 : 1];
  if (IDX && !to_state) {
    const uint4* wr = reinterpret_cast<const uint4*>(io.w_ik + size_t(t) * 512 + 128 * sg);
#pragma unroll
    for (int u8 = 0; u8 < (IDX ? 16 : 1); ++u8) wv[u8] = wr[u8];
  }
  // first token of this block's group (row of P); for from_state, the group's second token
  const size_t row0 = to_state ? size_t(b) * T + T - 1
                               : size_t(b) * T + (from_state ? 0 : head + size_t(r - head) * m);
  // channels 4t..4t+3 of up to m = 2 rows, projection (kv) and gate (z) halves:
  // vectors kv0 z0 kv1 z1 (m = 1: kv0 only)
  int v_lo = 0, v_hi = m == 1 ? 1 : 4;
  size_t off[4];
  off[0] = row0 * Nout + 4 * t;
  off[1] = row0 * Nout + 512 + 4 * t;
  off[2] = (row0 + 1) * Nout + 4 * t;
  off[3] = (row0 + 1) * Nout + 512 + 4 * t;
  if (to_state) {
    v_hi = 2;
  } else if (from_state) {   // kv1 z1 from row 0; kv0 z0 from the tail row, if any
    v_lo = stash_too ? 0 : 2;
    off[2] = off[0];
    off[3] = off[1];
    off[0] = (size_t(b) * T + T - 1) * Nout + 4 * t;
    off[1] = off[0] + 512;
  }
  const int sp0 = sg * n_split / 4, sp1 = (sg + 1) * n_split / 4;
  float4 acc[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = sp0; base < sp1; base += 4) {
    float4 ld[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int v = 0; v < 4; ++v)
        ld[q][v] = (base + q < sp1 && v >= v_lo && v < v_hi)
                       ? *reinterpret_cast<const float4*>(P + off[v] + size_t(base + q) * split_stride)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        if (base + q >= sp1 || v < v_lo || v >= v_hi) continue;
        acc[v].x += ld[q][v].x; acc[v].y += ld[q][v].y; acc[v].z += ld[q][v].z; acc[v].w += ld[q][v].w;
      }
  }
  if (sg > 0) {
#pragma unroll
    for (int v = 0; v < 4; ++v) part[sg - 1][t][v] = acc[v];
  }
  __syncthreads();
  if (IDX && !to_state && sg > 0) {   // groups 1..3: the key projection once the entry is in ys
    __syncthreads();
    idx_quarter(ys, wv, sg, t, ipart);
    return;
  }
  if (sg > 0) return;   // the rest runs in group 0 (4 warps)
#pragma unroll
  for (int q = 0; q < 3; ++q)
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const float4 o = part[q][t][v];
      acc[v].x += o.x; acc[v].y += o.y; acc[v].z += o.z; acc[v].w += o.w;
    }
  if (to_state) {
    *reinterpret_cast<float4*>(state + size_t(b) * 1024 + 4 * t) = acc[0];
    *reinterpret_cast<float4*>(state + size_t(b) * 1024 + 512 + 4 * t) = acc[1];
    return;
  }
  if (from_state) {
    float4* sp = reinterpret_cast<float4*>(state + size_t(b) * 1024 + 4 * t);
    const float4 k0 = sp[0], z0 = sp[128];
    if (stash_too) {
      sp[0] = acc[0];
      sp[128] = acc[1];
    }
    acc[0] = k0;
    acc[1] = z0;
  }
  float pooled[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    auto comp = [&](const float4& x) { return u == 0 ? x.x : u == 1 ? x.y : u == 2 ? x.z : x.w; };
    if (m == 1) {
      pooled[u] = comp(acc[0]);
    } else {
      const float kvv[2] = {comp(acc[0]), comp(acc[2])}, zz[2] = {comp(acc[1]), comp(acc[3])};
      const float mx = fmaxf(zz[0], zz[1]);
      float num = 0.f, den = 0.f;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float w = expf(zz[i] - mx);
        den += w;
        num = fmaf(w, kvv[i], num);
      }
      pooled[u] = num / den;
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int u = 0; u < 4; ++u) ss = fmaf(pooled[u], pooled[u], ss);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  __shared__ float red[4];
  if ((t & 31) == 0) red[t >> 5] = ss;
  asm volatile("bar.sync 1, 128;" ::: "memory");
  const float tot = (red[0] + red[1]) + (red[2] + red[3]);
  const float inv = 1.0f / sqrtf(tot / 512.0f + eps);
  float y[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) y[u] = norm_w[4 * t + u] * (pooled[u] * inv);
  if (kv_pre) {
    float4 v = make_float4(y[0], y[1], y[2], y[3]);
    *reinterpret_cast<float4*>(kv_pre + (size_t(b) * n_ent + r) * 512 + 4 * t) = v;
  }
  if (IDX) *reinterpret_cast<float4*>(&ys[4 * t]) = make_float4(y[0], y[1], y[2], y[3]);
  if (4 * t >= 448) {
    const long long pos = (long long)(pos0 / m + r) * m;   // the group's first token
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      const int i = (4 * t - 448) / 2 + pr;
      float c, s;
      rope_cs(pos, i, rt, c, s);
      const float a = y[2 * pr], bb = y[2 * pr + 1];
      y[2 * pr] = a * c - bb * s;
      y[2 * pr + 1] = a * s + bb * c;
    }
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(y[0], y[1]);
  __nv_bfloat162 hi = __floats2bfloat162_rn(y[2], y[3]);
  uint2 st;
  st.x = *reinterpret_cast<uint32_t*>(&lo);
  st.y = *reinterpret_cast<uint32_t*>(&hi);
  const size_t crow = size_t(b) * n_cap + size_t(pos0 / m) + r;
  *reinterpret_cast<uint2*>(kv_cache + crow * 512 + 4 * t) = st;
  if (IDX) {
    __syncthreads();   // ys complete (groups 1..3 wait here too)
    float acc_k = idx_quarter(ys, wv, 0, t, ipart);
    acc_k = ((acc_k + ipart[0][t]) + ipart[1][t]) + ipart[2][t];
    idx_finish(acc_k, t, (long long)(pos0 / m + r), m, rt, io.codes, io.scales, crow, nullptr, 0);
  }
}

constexpr int IK_E = 8;  // entries per block (few entries, as in decode: 2)

// 512 threads: thread j + 128 qk computes key dim j for E entries over inputs 128 qk ..
// 128 qk + 127 (its 16 weight loads in flight together); the four quarter sums are added in
// quarter order (deterministic), then warp w of the first 128 threads quantises block w
// (dims 32w..32w+31) of each entry.
template <int E>
__global__ void __launch_bounds__(512) index_k_kernel(const float* __restrict__ kv_pre, int B,
                                                      int G, int entry0, int m,
                                                      const uint16_t* __restrict__ w_ik,
                                                      const RopeTurns rt, uint8_t* __restrict__ codes,
                                                      uint8_t* __restrict__ scales, int n_cap,
                                                      float* __restrict__ k_out) {
  pdl_wait();
  __shared__ float kv[E][512];
  __shared__ float part[3][E][128];
  const int tid = threadIdx.x, j = tid & 127, qk = tid >> 7;
  const int total = B * G;
  const int e0 = blockIdx.x * E;
  for (int idx = tid * 4; idx < E * 512; idx += 512 * 4) {
    const int e = e0 + idx / 512;
    *reinterpret_cast<float4*>(&kv[idx / 512][idx % 512]) =
        (e < total) ? *reinterpret_cast<const float4*>(kv_pre + size_t(e) * 512 + idx % 512)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  uint4 vv[16];
  const uint4* wr = reinterpret_cast<const uint4*>(w_ik + size_t(j) * 512 + 128 * qk);
#pragma unroll
  for (int u8 = 0; u8 < 16; ++u8) vv[u8] = wr[u8];
  __syncthreads();
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
  for (int u8 = 0; u8 < 16; ++u8) {
    const uint16_t* pv = reinterpret_cast<const uint16_t*>(&vv[u8]);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float wv = bf16_to_f32(pv[u]);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(wv, kv[e][128 * qk + 8 * u8 + u], acc[e]);
    }
  }
  if (qk > 0) {
#pragma unroll
    for (int e = 0; e < E; ++e) part[qk - 1][e][j] = acc[e];
  }
  __syncthreads();
  if (qk > 0) return;   // the rest runs in the first 128 threads
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = ((acc[e] + part[0][e][j]) + part[1][e][j]) + part[2][e][j];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int ei = e0 + e;
    if (ei >= total) break;  // uniform across the block
    const int b = ei / G, g = ei % G;
    const long long ent = (long long)entry0 + g;
    idx_finish(acc[e], j, ent, m, rt, codes, scales, size_t(b) * n_cap + size_t(ent), k_out, size_t(ei));
  }
}

// FP8 window-KV rows: one warp per row, lane l owns channels 16 l .. 16 l + 15; four lanes
// form a 64-channel scale group.  Scale 2^k with k = fp8_scale_exp(group amax) (stored as
// k + 127), codes sign << 7 | E4M3 nearest-even of |v| * 2^-k (an exact product).
__global__ void __launch_bounds__(256) swa_kv_fp8_kernel(const uint16_t* __restrict__ swa, int B,
                                                         int S, int row0, int n_rows,
                                                         uint8_t* __restrict__ codes,
                                                         uint8_t* __restrict__ scales) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long e = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (e >= (long long)B * n_rows) return;   // whole warps leave together
  const long long b = e / n_rows, r = e % n_rows;
  const size_t row = size_t(b) * S + size_t(row0 + r);
  const uint4* src = reinterpret_cast<const uint4*>(swa + row * 512 + 16 * lane);
  const uint4 w0 = src[0], w1 = src[1];
  const uint32_t wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  float v[16];
  float amax = 0.f;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    v[2 * u] = __uint_as_float(wd[u] << 16);
    v[2 * u + 1] = __uint_as_float(wd[u] & 0xFFFF0000u);
    amax = fmaxf(amax, fmaxf(fabsf(v[2 * u]), fabsf(v[2 * u + 1])));
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const int k = fp8_scale_exp(amax);
  const float inv = __uint_as_float(uint32_t(127 - k) << 23);   // 2^-k, k in [-126, 120]
  uint32_t out[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const float q = v[u] * inv;
    const uint32_t c = ((__float_as_uint(q) >> 31) << 7) | e4m3_rne_satfinite(fabsf(q));
    out[u >> 2] |= c << (8 * (u & 3));
  }
  *reinterpret_cast<uint4*>(codes + row * 512 + 16 * lane) = make_uint4(out[0], out[1], out[2], out[3]);
  if ((lane & 3) == 0) scales[row * 8 + (lane >> 2)] = uint8_t(k + 127);
}

// FP4 main-KV entries: one warp per entry, lane l owns channels 16 l .. 16 l + 15 (one
// scale group): E4M3 scale = nearest-even(amax / 6) saturating, E2M1 codes nearest-even of
// v / scale (float32 divides), element 2 i in the low nibble of byte i.
__global__ void __launch_bounds__(256) main_kv_fp4_kernel(const uint16_t* __restrict__ kv, int B,
                                                          int n_cap, int entry0, int G,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long e = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (e >= (long long)B * G) return;
  const long long b = e / G, g = e % G;
  const size_t row = size_t(b) * n_cap + size_t(entry0 + g);
  const uint4* src = reinterpret_cast<const uint4*>(kv + row * 512 + 16 * lane);
  const uint4 w0 = src[0], w1 = src[1];
  const uint32_t wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  float v[16];
  float amax = 0.f;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    v[2 * u] = __uint_as_float(wd[u] << 16);
    v[2 * u + 1] = __uint_as_float(wd[u] & 0xFFFF0000u);
    amax = fmaxf(amax, fmaxf(fabsf(v[2 * u]), fabsf(v[2 * u + 1])));
  }
  const uint32_t sb = e4m3_rne_satfinite(__fdiv_rn(amax, 6.0f));
  uint32_t packed[2] = {0u, 0u};
  if (sb != 0u) {
    const float sc = e4m3_value(sb);
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const float q = __fdiv_rn(v[u], sc);
      const uint32_t c = ((__float_as_uint(q) >> 31) << 3) | e2m1_rne_mag(fabsf(q));
      packed[u >> 3] |= c << (4 * (u & 7));
    }
  }
  *reinterpret_cast<uint2*>(codes + row * 256 + 8 * lane) = make_uint2(packed[0], packed[1]);
  scales[row * 32 + lane] = uint8_t(sb);
}

}  // namespace
}  // namespace csa2

using namespace csa2;

namespace {

// Shared body of the compressor entry points: tokens pos0 .. pos0+T-1 of B sequences, any
// pos0 when `state` is given (m = 2), else pos0 % m == 0 and a trailing partial group ignored.
// With idx (the runner's Full layers), a call of at most IDX_FUSE_ENTRIES entries also writes
// their indexer keys from the epilogue (*fused = true); otherwise the caller runs the
// indexer-key kernel on kv_pre.
constexpr long long IDX_FUSE_ENTRIES = 4096;
int compress_impl(const char* who, const void* x, int B, int T, int hidden, int m, int pos0,
                  const void* w_kv, const void* w_gate, const float* norm_w, float eps,
                  float rope_base, float* state, void* kv_cache, int n_cap, float* kv_pre,
                  void* workspace, size_t ws_bytes, void* stream, const IdxOut* idx = nullptr,
                  bool* fused = nullptr) {
  if (fused) *fused = false;
  if (m != 1 && m != 2) return fail(CSA2_ERR_UNSUPPORTED, "%s: m must be 1 or 2 (got %d)", who, m);
  if (!x || !w_kv || !norm_w || !kv_cache)
    return fail(CSA2_ERR_INVALID_ARG, "%s: null tensor pointer", who);
  if ((m == 1) != (w_gate == nullptr))
    return fail(CSA2_ERR_INVALID_ARG, "%s: w_gate must be NULL exactly when m == 1", who);
  if (B <= 0 || T <= 0 || hidden <= 0 || hidden % 64 != 0)
    return fail(CSA2_ERR_INVALID_ARG, "%s: bad shape B=%d T=%d hidden=%d", who, B, T, hidden);
  if (pos0 < 0 || (!state && pos0 % m != 0))
    return fail(CSA2_ERR_INVALID_ARG, "%s: pos0=%d must be >= 0 and a multiple of m", who, pos0);
  const int head = (state && pos0 % m != 0) ? 1 : 0;
  const int tail = (state && ((long long)pos0 + T) % m != 0) ? 1 : 0;
  const int n_ent = state ? int(((long long)pos0 + T) / m - pos0 / m) : T / m;
  if (n_cap <= 0 || (long long)pos0 / m + n_ent > n_cap)
    return fail(CSA2_ERR_INVALID_ARG, "%s: entries %d..%d exceed n_cap=%d", who, pos0 / m,
                pos0 / m + n_ent - 1, n_cap);
  if (!(eps >= 0.f) || !(rope_base > 0.f))
    return fail(CSA2_ERR_INVALID_ARG, "%s: bad eps / rope_base", who);
  if (!aligned16(x) || !aligned16(w_kv) || (w_gate && !aligned16(w_gate)) || !aligned16(norm_w) ||
      !aligned16(kv_cache) || (kv_pre && !aligned16(kv_pre)) || (state && !aligned16(state)))
    return fail(CSA2_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", who);
  if ((long long)B * T > (1ll << 30))
    return fail(CSA2_ERR_UNSUPPORTED, "%s: B*T too large for one call", who);
  const size_t need = csa2_compress_workspace_size(B, T, hidden, m);
  if (!workspace || ws_bytes < need || !aligned256(workspace))
    return fail(CSA2_ERR_WORKSPACE, "%s: workspace needs %zu bytes, 256-aligned", who, need);
  if (idx && (!idx->w_ik || !idx->codes || !idx->scales || !aligned16(idx->w_ik)))
    return fail(CSA2_ERR_INVALID_ARG, "%s: indexer-key weights and caches needed, 16-byte aligned", who);
  if (n_ent + tail == 0) return CSA2_OK;   // (n_ent == 0 implies head == 0)
  cudaStream_t st = (cudaStream_t)stream;
  const int M = B * T, nout = (m == 1) ? 512 : 1024;
  float* P = static_cast<float*>(workspace);
  int splits = 1;
  if (hidden % 256 == 0) {
    splits = proj_splits(M, hidden, nout);
    cudaError_t e0 = cudaFuncSetAttribute(proj_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          int(PU_SMEM));
    if (e0 != cudaSuccess) return cuda_fail(e0, "compress: shared memory attribute");
    // operand tensor maps: [rows][hidden] bf16, boxes of 64 elements (128 bytes) x 128 rows
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return fail(CSA2_ERR_CUDA, "%s: cuTensorMapEncodeTiled not available", who);
    auto make_map = [&](CUtensorMap* map, const void* ptr, long long rows_) -> bool {
      const cuuint64_t dims[2] = {cuuint64_t(hidden), cuuint64_t(rows_)};
      const cuuint64_t strides[1] = {cuuint64_t(hidden) * 2};
      const cuuint32_t box[2] = {cuuint32_t(PU_KC), cuuint32_t(PU_TILE)};
      const cuuint32_t estr[2] = {1, 1};
      return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    CUtensorMap x_map, w0_map, w1_map;
    if (!make_map(&x_map, x, M) || !make_map(&w0_map, w_kv, 512) ||
        !make_map(&w1_map, w_gate ? w_gate : w_kv, 512))
      return fail(CSA2_ERR_CUDA, "%s: operand tensor maps", who);
    dim3 grid(nout / PU_TILE, ceil_div(M, PU_TILE), splits);
    CSA2_LAUNCH("proj_umma launch", proj_umma_kernel, grid, PU_T, PU_SMEM, st, x_map, w0_map, w1_map, M, nout, hidden / splits, P);
  } else {
    dim3 grid(nout / GN, ceil_div(M, GM));
    CSA2_LAUNCH("proj_gemm launch", proj_gemm_kernel, grid, GT, 0, st, (const uint16_t*)x, (const uint16_t*)w_kv, (const uint16_t*)w_gate, M, hidden, nout, P);
  }
  note_launch();
  const bool use_idx = idx && (long long)B * n_ent <= IDX_FUSE_ENTRIES;
  const unsigned n_blocks = unsigned(B * (n_ent + (tail && !head ? 1 : 0)));
  if (use_idx) {
    CSA2_LAUNCH("compress_epilogue launch", compress_epilogue_kernel<true>, n_blocks, 512, 0, st, P, splits, size_t(M) * nout, nout, T, m, pos0, n_ent, head, tail, norm_w, eps, rope_turns(rope_base), (uint16_t*)kv_cache, n_cap, kv_pre, state, *idx);
  } else {
    CSA2_LAUNCH("compress_epilogue launch", compress_epilogue_kernel<false>, n_blocks, 512, 0, st, P, splits, size_t(M) * nout, nout, T, m, pos0, n_ent, head, tail, norm_w, eps, rope_turns(rope_base), (uint16_t*)kv_cache, n_cap, kv_pre, state, IdxOut{nullptr, nullptr, nullptr});
  }
  note_launch();
  if (fused) *fused = use_idx;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "compress launch");
  return CSA2_OK;
}

}  // namespace

int csa2::compress_index_k(const void* x, int B, int T, int hidden, int m, int pos0, const void* w_kv,
                           const void* w_gate, const float* norm_w, float eps, float rope_base,
                           float* state, void* kv_cache, int n_cap, float* kv_pre, void* workspace,
                           size_t ws_bytes, const void* w_ik, uint8_t* idx_codes, uint8_t* idx_scales,
                           void* stream, bool* fused) {
  if (fused) *fused = false;
  if (m == 1 && state) return fail(CSA2_ERR_INVALID_ARG, "compress_chunk: state must be NULL when m == 1");
  const IdxOut io{static_cast<const uint16_t*>(w_ik), idx_codes, idx_scales};
  return compress_impl(state ? "compress_chunk" : "compress", x, B, T, hidden, m, pos0, w_kv, w_gate,
                       norm_w, eps, rope_base, state, kv_cache, n_cap, kv_pre, workspace, ws_bytes,
                       stream, &io, fused);
}

extern "C" {

size_t csa2_compress_workspace_size(int B, int T, int hidden, int m) {
  if (B <= 0 || T <= 0 || (m != 1 && m != 2) || hidden <= 0) return 0;
  const int nout = (m == 1) ? 512 : 1024;
  const long long M = (long long)B * T;
  const int splits = (hidden % 256 == 0 && M <= (1ll << 30)) ? proj_splits(int(M), hidden, nout) : 1;
  return align_up(size_t(splits) * size_t(M) * nout * sizeof(float), 256);
}

int csa2_compress(const void* x, int B, int T, int hidden, int m, int pos0, const void* w_kv,
                  const void* w_gate, const float* norm_w, float eps, float rope_base,
                  void* kv_cache, int n_cap, float* kv_pre, void* workspace, size_t ws_bytes,
                  void* stream) {
  return compress_impl("compress", x, B, T, hidden, m, pos0, w_kv, w_gate, norm_w, eps, rope_base,
                       nullptr, kv_cache, n_cap, kv_pre, workspace, ws_bytes, stream);
}

int csa2_compress_chunk(const void* x, int B, int T, int hidden, int m, int pos0, const void* w_kv,
                        const void* w_gate, const float* norm_w, float eps, float rope_base,
                        float* state, void* kv_cache, int n_cap, float* kv_pre, void* workspace,
                        size_t ws_bytes, void* stream) {
  if (m == 2 && !state) return fail(CSA2_ERR_INVALID_ARG, "compress_chunk: m == 2 needs a state buffer");
  if (m == 1 && state) return fail(CSA2_ERR_INVALID_ARG, "compress_chunk: state must be NULL when m == 1");
  return compress_impl("compress_chunk", x, B, T, hidden, m, pos0, w_kv, w_gate, norm_w, eps,
                       rope_base, state, kv_cache, n_cap, kv_pre, workspace, ws_bytes, stream);
}

int csa2_index_k_quant(const float* kv_pre, int B, int G, int entry0, int m, const void* w_ik,
                       float rope_base, uint8_t* codes, uint8_t* scales, int n_cap, float* k_out,
                       void* stream) {
  if (!kv_pre || !w_ik || !codes || !scales)
    return fail(CSA2_ERR_INVALID_ARG, "index_k_quant: null tensor pointer");
  if (B <= 0 || G < 0 || entry0 < 0 || m < 1 || n_cap <= 0 || (long long)entry0 + G > n_cap)
    return fail(CSA2_ERR_INVALID_ARG, "index_k_quant: bad shape B=%d G=%d entry0=%d n_cap=%d", B,
                G, entry0, n_cap);
  if (!(rope_base > 0.f)) return fail(CSA2_ERR_INVALID_ARG, "index_k_quant: bad rope_base");
  if (!aligned16(kv_pre) || !aligned16(w_ik) || !aligned16(codes) || !aligned16(scales) ||
      (k_out && !aligned16(k_out)))
    return fail(CSA2_ERR_INVALID_ARG, "index_k_quant: pointers must be 16-byte aligned");
  if ((long long)B * G > (1ll << 31) - IK_E)
    return fail(CSA2_ERR_UNSUPPORTED, "index_k_quant: too many entries for one call");
  if (G == 0) return CSA2_OK;
  const int total = B * G;
  if (total <= 1024) {   // few entries (decode): more CTAs, each reading the weights once
    CSA2_LAUNCH("index_k launch", index_k_kernel<2>, ceil_div(total, 2), 512, 0, (cudaStream_t)stream, kv_pre, B, G, entry0, m, (const uint16_t*)w_ik, rope_turns(rope_base), codes, scales, n_cap, k_out);
  } else {
    CSA2_LAUNCH("index_k launch", index_k_kernel<IK_E>, ceil_div(total, IK_E), 512, 0, (cudaStream_t)stream, kv_pre, B, G, entry0, m, (const uint16_t*)w_ik, rope_turns(rope_base), codes, scales, n_cap, k_out);
  }
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "index_k_quant launch");
  return CSA2_OK;
}

int csa2_swa_kv_quant_fp8(const void* swa_kv, int B, int S, int row0, int n_rows,
                          uint8_t* codes, uint8_t* scales, void* stream) {
  if (!swa_kv || !codes || !scales)
    return fail(CSA2_ERR_INVALID_ARG, "swa_kv_quant_fp8: null tensor pointer");
  if (B <= 0 || n_rows < 0 || row0 < 0 || S <= 0 || (long long)row0 + n_rows > S)
    return fail(CSA2_ERR_INVALID_ARG, "swa_kv_quant_fp8: bad shape B=%d rows %d..+%d S=%d",
                B, row0, n_rows, S);
  if (!aligned16(swa_kv) || !aligned16(codes) || !aligned16(scales))
    return fail(CSA2_ERR_INVALID_ARG, "swa_kv_quant_fp8: pointers must be 16-byte aligned");
  if ((long long)B * n_rows > (1ll << 34))
    return fail(CSA2_ERR_UNSUPPORTED, "swa_kv_quant_fp8: too many rows for one call");
  if (n_rows == 0) return CSA2_OK;
  const long long blocks = ((long long)B * n_rows + 7) / 8;
  CSA2_LAUNCH("swa_kv_fp8 launch", swa_kv_fp8_kernel, unsigned(blocks), 256, 0, (cudaStream_t)stream,
              (const uint16_t*)swa_kv, B, S, row0, n_rows, codes, scales);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "swa_kv_quant_fp8 launch");
  return CSA2_OK;
}

int csa2_main_kv_quant_fp4(const void* kv_cache, int B, int n_cap, int entry0, int G,
                           uint8_t* codes, uint8_t* scales, void* stream) {
  if (!kv_cache || !codes || !scales)
    return fail(CSA2_ERR_INVALID_ARG, "main_kv_quant_fp4: null tensor pointer");
  if (B <= 0 || G < 0 || entry0 < 0 || n_cap <= 0 || (long long)entry0 + G > n_cap)
    return fail(CSA2_ERR_INVALID_ARG, "main_kv_quant_fp4: bad shape B=%d G=%d entry0=%d n_cap=%d",
                B, G, entry0, n_cap);
  if (!aligned16(kv_cache) || !aligned16(codes) || !aligned16(scales))
    return fail(CSA2_ERR_INVALID_ARG, "main_kv_quant_fp4: pointers must be 16-byte aligned");
  if ((long long)B * G > (1ll << 34))
    return fail(CSA2_ERR_UNSUPPORTED, "main_kv_quant_fp4: too many entries for one call");
  if (G == 0) return CSA2_OK;
  const long long blocks = ((long long)B * G + 7) / 8;
  CSA2_LAUNCH("main_kv_fp4 launch", main_kv_fp4_kernel, unsigned(blocks), 256, 0, (cudaStream_t)stream,
              (const uint16_t*)kv_cache, B, n_cap, entry0, G, codes, scales);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "main_kv_quant_fp4 launch");
  return CSA2_OK;
}

}  // extern "C"
