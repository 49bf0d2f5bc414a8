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
// attn_umma_kernel (64 heads): one CTA per (query row, tile of 128 rows of A).  The rows
// are gathered with 16-byte asynchronous copies into a K-major 128-byte-swizzled tile;
// tcgen05 computes S^T = C Q^T (128 rows x 64 heads, K = 512) into TMEM; each head's
// softmax over the tile's rows gives (max, sum) and P^T (bf16, MN-major); tcgen05 then
// computes O^T = C^T P^T (512 dims x 64 heads, K = 128 rows) reading the SAME shared
// tile as an MN-major operand (K = V).  attn_combine_kernel merges the per-tile
// (max, sum, O) partials of a row into the normalised output.
//
// attn_simt_kernel (any H): one CTA per (query row, group of 8 heads), one warp per head.
// Rows of A (top-k slots then window rows) stream through shared memory in tiles of
// 32; lane j scores row j of the tile; an online softmax keeps (max, sum) per head
// and every lane accumulates 16 of the 512 output dims.
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
};

__global__ void __launch_bounds__(AT_T) attn_simt_kernel(AttnArgs a) {
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


constexpr int AU_T = 256;            // threads
constexpr int AU_ROWS = 128;         // rows of A per CTA (M of the first MMA)
constexpr int AU_H = 64;             // heads (N of both MMAs)
constexpr uint32_t AU_KV_BYTES = AU_ROWS * 512 * 2;    // 128 KB
constexpr uint32_t AU_Q_BYTES = AU_H * 512 * 2;        // 64 KB (reused for S^T in f32)
constexpr uint32_t AU_P_BYTES = AU_ROWS * AU_H * 2;    // 16 KB
constexpr uint32_t AU_SMEM = AU_KV_BYTES + AU_Q_BYTES + AU_P_BYTES + 1024;

struct AttnUmmaArgs {
  AttnArgs a;
  int n_tiles;
  float* part_o;    // [rows][n_tiles][64][512]
  float* part_ml;   // [rows][n_tiles][64][2]
};

__global__ void __launch_bounds__(AU_T, 1) attn_umma_kernel(AttnUmmaArgs u) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* KV = base;
  uint8_t* Qs = base + AU_KV_BYTES;
  float* Sbuf = reinterpret_cast<float*>(Qs);          // [64][128] after the first MMA
  uint8_t* Ps = base + AU_KV_BYTES + AU_Q_BYTES;
  __shared__ const uint16_t* row_src[AU_ROWS];
  __shared__ int row_ok[AU_ROWS];
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int any_valid;

  const AttnArgs& a = u.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = blockIdx.x / u.n_tiles, tile = blockIdx.x % u.n_tiles;
  const int b = row / a.Tq, i = row % a.Tq;
  const long long t = (long long)a.q_pos0 + i;
  const long long lo = t - a.window + 1 > 0 ? t - a.window + 1 : 0;
  const int n_rows = a.k + int(t - lo + 1);
  float* ml = u.part_ml + (size_t(row) * u.n_tiles + tile) * AU_H * 2;

  if (tid == 0) any_valid = 0;
  __syncthreads();
  if (tid < AU_ROWS) {
    const int j = tile * AU_ROWS + tid;
    int ok = 0;
    const uint16_t* src = a.swa;   // any valid address for zero-filled copies
    if (j < a.k) {
      const int e = a.topk[size_t(row) * a.k + j];
      if (e >= a.n_entries) atomicOr(&d_err_attn, ERR_BOUNDS);
      if (e >= 0 && e < a.n_entries) {
        ok = 1;
        src = a.kv + (size_t(b) * a.n_cap + e) * 512;
      }
    } else if (j < n_rows) {
      ok = 1;
      src = a.swa + (size_t(b) * a.S + size_t(lo + (j - a.k) - a.swa_pos0)) * 512;
    }
    row_src[tid] = src;
    row_ok[tid] = ok;
    if (ok) atomicOr(&any_valid, 1);
  }
  __syncthreads();
  if (!any_valid) {          // tile entirely past this row's set: empty partial
    if (tid < AU_H) { ml[2 * tid] = -INFINITY; ml[2 * tid + 1] = 0.f; }
    return;
  }
  if (tid == 0) {
    umma::mbar_init(&bar[0], 1);
    umma::mbar_init(&bar[1], 1);
    umma::mbar_fence_init();
  }
  if (warp == 0) umma::tmem_alloc(&tmem_slot, 512);

  // gather, one commit group per 64-dim atom column: 128 rows x 8 chunks of the KV tile
  // and 64 heads x 8 chunks of the query block; the first MMA consumes atom a as soon
  // as every thread's group a has landed.
  const uint16_t* qrow = a.q + size_t(row) * a.H * 512;
#pragma unroll 1
  for (int at = 0; at < 8; ++at) {
    for (int c = tid; c < AU_ROWS * 8; c += AU_T) {
      const int r = c >> 3, ch = at * 8 + (c & 7);
      umma::cp_async16(KV + umma::kmajor_sw128_offset(r, ch * 8, AU_ROWS), row_src[r] + ch * 8,
                       row_ok[r] ? 16u : 0u);
    }
    for (int c = tid; c < AU_H * 8; c += AU_T) {
      const int h = c >> 3, ch = at * 8 + (c & 7);
      umma::cp_async16(Qs + umma::kmajor_sw128_offset(h, ch * 8, AU_H), qrow + h * 512 + ch * 8, 16u);
    }
    umma::cp_async_commit();
  }
  uint32_t tmem = 0;
  constexpr uint32_t idesc_s = umma::idesc_f16(AU_ROWS, AU_H, 1, 0, 0);
  const uint32_t kv_base = umma::smem_u32(KV), q_base = umma::smem_u32(Qs);
#pragma unroll
  for (int at = 0; at < 8; ++at) {
    umma::cp_async_wait_pending(7 - at);
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    if (at == 0) tmem = tmem_slot;
    // S^T = C Q^T over dims 64*at .. 64*at + 63 (4 steps of K = 16)
    if (tid == 0) {
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const uint64_t da = umma::desc_sw128(kv_base + at * (AU_ROWS * 128) + k4 * 32, 16, 1024);
        const uint64_t db = umma::desc_sw128(q_base + at * (AU_H * 128) + k4 * 32, 16, 1024);
        umma::mma_f16(tmem, da, db, idesc_s, (at | k4) != 0);
      }
      if (at == 7) umma::commit(&bar[0]);
    }
  }
  // logits are kept in base-2 units (scaled by log2 e) so the softmax uses exp2;
  // (max, sum) partials are converted back to natural units for the combine.
  const float scale_log2 = a.scale * 1.4426950408889634f;
  bool ok = true;
  ok = umma::mbar_wait(&bar[0], 0, &d_err_attn);
  umma::fence_after();
  if (ok) {
    const int q = warp & 3, half = warp >> 2;
    const int r = q * 32 + lane;
    const bool valid = row_ok[r] != 0;
    uint32_t v[32];
    umma::tmem_ld32(tmem + (uint32_t(q * 32) << 16) + uint32_t(half * 32), v);
    umma::tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < 32; ++h)
      Sbuf[(half * 32 + h) * AU_ROWS + r] = valid ? __uint_as_float(v[h]) * scale_log2 : -INFINITY;
  }
  umma::fence_before();
  __syncthreads();
  umma::fence_after();

  // softmax within the tile: warp w owns heads 8w .. 8w+7, lane owns rows lane + 32 j;
  // P^T row r gets the 8 heads' probabilities as one 16-byte chunk.
  {
    const int h0 = warp * 8;
    float p[4][8];
#pragma unroll
    for (int hh = 0; hh < 8; ++hh) {
      const float* srow = Sbuf + (h0 + hh) * AU_ROWS + lane;
      float v0 = srow[0], v1 = srow[32], v2 = srow[64], v3 = srow[96];
      float m = fmaxf(fmaxf(v0, v1), fmaxf(v2, v3));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const bool live = m != -INFINITY;
      p[0][hh] = live ? exp2f(v0 - m) : 0.f;
      p[1][hh] = live ? exp2f(v1 - m) : 0.f;
      p[2][hh] = live ? exp2f(v2 - m) : 0.f;
      p[3][hh] = live ? exp2f(v3 - m) : 0.f;
      float l = (p[0][hh] + p[1][hh]) + (p[2][hh] + p[3][hh]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (lane == 0) { ml[2 * (h0 + hh)] = m * 0.6931471805599453f; ml[2 * (h0 + hh) + 1] = l; }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = lane + 32 * j;
      uint32_t w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        __nv_bfloat162 v2 = __floats2bfloat162_rn(p[j][2 * u], p[j][2 * u + 1]);
        w[u] = *reinterpret_cast<uint32_t*>(&v2);
      }
      const uint32_t off = uint32_t((r >> 3) * 1024 + (r & 7) * 128 + ((warp ^ (r & 7)) << 4));
      *reinterpret_cast<uint4*>(Ps + off) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  umma::fence_proxy_async();
  umma::fence_before();
  __syncthreads();
  umma::fence_after();

  // O^T = C^T P^T: four 128-dim tiles, 8 steps of K = 16 rows
  if (tid == 0 && ok) {
    constexpr uint32_t idesc = umma::idesc_f16(128, AU_H, 1, 1, 1);
    const uint32_t kv0 = umma::smem_u32(KV), p0 = umma::smem_u32(Ps);
    for (int dt = 0; dt < 4; ++dt)
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t da = umma::desc_sw128(kv0 + (2 * dt) * (AU_ROWS * 128) + kk * 2048,
                                             AU_ROWS * 128, 1024);
        const uint64_t db = umma::desc_sw128(p0 + kk * 2048, AU_ROWS * 128, 1024);
        umma::mma_f16(tmem + 64 + 64 * dt, da, db, idesc, kk > 0);
      }
    umma::commit(&bar[1]);
  }
  if (ok) ok = umma::mbar_wait(&bar[1], 0, &d_err_attn);
  umma::fence_after();
  if (ok) {
    const int q = warp & 3;
    float* po = u.part_o + (size_t(row) * u.n_tiles + tile) * AU_H * 512;
#pragma unroll 1
    for (int dti = 0; dti < 2; ++dti) {
      const int dt = (warp >> 2) * 2 + dti;
      const int d = dt * 128 + q * 32 + lane;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t v[32];
        umma::tmem_ld32(tmem + (uint32_t(q * 32) << 16) + uint32_t(64 + 64 * dt + 32 * half), v);
        umma::tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < 32; ++h) po[size_t(half * 32 + h) * 512 + d] = __uint_as_float(v[h]);
      }
    }
  }
  umma::fence_before();
  __syncthreads();
  if (warp == 0) umma::tmem_free(tmem, 512);
}

// One CTA per (query row, group of 8 heads), 128 threads: thread t owns dims 4t..4t+3.
// All tile partials of a head are loaded before they are combined so that the loads
// are in flight together.
constexpr int AC_HG = 8;
__global__ void __launch_bounds__(128) attn_combine_kernel(AttnUmmaArgs u) {
  const AttnArgs& a = u.a;
  __shared__ float wgt[AC_HG][8];    // per head, per tile: e^(m_t - M) / L (0 if empty)
  const int row = blockIdx.x / (AU_H / AC_HG), hg = blockIdx.x % (AU_H / AC_HG);
  const int tid = threadIdx.x;
  const float* __restrict__ ml = u.part_ml + size_t(row) * u.n_tiles * AU_H * 2;
  if (tid < AC_HG) {
    const int h = hg * AC_HG + tid;
    float M = -INFINITY;
    for (int tt = 0; tt < u.n_tiles; ++tt)
      if (ml[(tt * AU_H + h) * 2 + 1] > 0.f) M = fmaxf(M, ml[(tt * AU_H + h) * 2]);
    if (a.sink) M = fmaxf(M, a.sink[h]);
    float L = 0.f;
    for (int tt = 0; tt < u.n_tiles; ++tt) {
      const float l = ml[(tt * AU_H + h) * 2 + 1];
      if (l > 0.f) L += l * expf(ml[(tt * AU_H + h) * 2] - M);
    }
    if (a.sink) L += expf(a.sink[h] - M);
    for (int tt = 0; tt < 8; ++tt) {
      float wv = 0.f;
      if (tt < u.n_tiles) {
        const float l = ml[(tt * AU_H + h) * 2 + 1];
        if (l > 0.f) wv = expf(ml[(tt * AU_H + h) * 2] - M) / L;
      }
      wgt[tid][tt] = wv;
    }
    if (a.lse) a.lse[size_t(row) * AU_H + h] = M + logf(L);
  }
  __syncthreads();
  const float4* __restrict__ po =
      reinterpret_cast<const float4*>(u.part_o + size_t(row) * u.n_tiles * AU_H * 512);
  __nv_bfloat16* __restrict__ out = reinterpret_cast<__nv_bfloat16*>(a.out);
#pragma unroll 1
  for (int hh = 0; hh < AC_HG; ++hh) {
    const int h = hg * AC_HG + hh;
    float4 v[8];
#pragma unroll
    for (int tt = 0; tt < 8; ++tt)
      v[tt] = (wgt[hh][tt] != 0.f) ? po[(size_t(tt) * AU_H + h) * 128 + tid] : make_float4(0, 0, 0, 0);
    float4 acc = make_float4(0, 0, 0, 0);
#pragma unroll
    for (int tt = 0; tt < 8; ++tt) {
      const float wv = wgt[hh][tt];
      acc.x = fmaf(wv, v[tt].x, acc.x); acc.y = fmaf(wv, v[tt].y, acc.y);
      acc.z = fmaf(wv, v[tt].z, acc.z); acc.w = fmaf(wv, v[tt].w, acc.w);
    }
    __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x, acc.y), hi2 = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 st;
    st.x = *reinterpret_cast<uint32_t*>(&lo2);
    st.y = *reinterpret_cast<uint32_t*>(&hi2);
    *reinterpret_cast<uint2*>(out + (size_t(row) * AU_H + h) * 512 + 4 * tid) = st;
  }
}

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" {

size_t csa2_sparse_attn_workspace_size(int B, int Tq, int H, int k, int window) {
  if (H != AU_H || B <= 0 || Tq <= 0 || k < 0 || window < 1) return 0;
  const size_t n_tiles = size_t(ceil_div(k + window, AU_ROWS));
  const size_t rows = size_t(B) * Tq;
  return align_up(rows * n_tiles * AU_H * 512 * sizeof(float), 256) +
         align_up(rows * n_tiles * AU_H * 2 * sizeof(float), 256);
}

int csa2_sparse_attn(const void* q, int B, int Tq, int H, int q_pos0, const void* kv_cache,
                     int n_cap, int n_entries, const int32_t* topk, int k, const void* swa_kv,
                     int S, int swa_pos0, int window, const float* sink, float scale, void* out,
                     float* lse_out, void* workspace, size_t ws_bytes, void* stream) {
  if (!q || !swa_kv || !out) return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: null tensor pointer");
  if (k < 0 || k > CSA2_MAX_TOPK) return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: k=%d out of [0, 2048]", k);
  if (k > 0 && (!topk || !kv_cache))
    return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: k > 0 needs topk and kv_cache");
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
      !aligned16(swa_kv) || !aligned16(out) || (sink && !aligned16(sink)) ||
      (lse_out && !aligned16(lse_out)))
    return fail(CSA2_ERR_INVALID_ARG, "sparse_attn: pointers must be 16-byte aligned");
  const long long rows = (long long)B * Tq;
  const int n_hg = ceil_div(H, AT_HG);
  if (rows * n_hg > (1ll << 31) - 1) return fail(CSA2_ERR_UNSUPPORTED, "sparse_attn: too many rows");
  AttnArgs aa{(const uint16_t*)q, int(rows), Tq, H, q_pos0, n_hg, (const uint16_t*)kv_cache,
              n_cap, n_entries, topk, k, (const uint16_t*)swa_kv, S, swa_pos0, window, sink,
              scale, (uint16_t*)out, lse_out};
  cudaStream_t st = (cudaStream_t)stream;
  if (H == AU_H) {
    // tensor-core path: per-tile partials in the workspace, then the combine
    const size_t need = csa2_sparse_attn_workspace_size(B, Tq, H, k, window);
    if (!workspace || ws_bytes < need || !aligned256(workspace))
      return fail(CSA2_ERR_WORKSPACE, "sparse_attn: workspace needs %zu bytes, 256-aligned", need);
    const int n_tiles = ceil_div(k + window, AU_ROWS);
    if (n_tiles > 8) return fail(CSA2_ERR_UNSUPPORTED, "sparse_attn: k + window > 1024 with 64 heads");
    if (rows * n_tiles > (1ll << 31) - 1) return fail(CSA2_ERR_UNSUPPORTED, "sparse_attn: too many rows");
    AttnUmmaArgs ua{aa, n_tiles, static_cast<float*>(workspace), nullptr};
    ua.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                          align_up(size_t(rows) * n_tiles * AU_H * 512 * 4, 256));
    cudaError_t e0 = cudaFuncSetAttribute(attn_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          int(AU_SMEM));
    if (e0 != cudaSuccess) return cuda_fail(e0, "sparse_attn: shared memory attribute");
    attn_umma_kernel<<<unsigned(rows * n_tiles), AU_T, AU_SMEM, st>>>(ua);
    note_launch();
    attn_combine_kernel<<<unsigned(rows * (AU_H / AC_HG)), 128, 0, st>>>(ua);
    note_launch();
  } else {
    attn_simt_kernel<<<unsigned(rows * n_hg), AT_T, 0, st>>>(aa);
    note_launch();
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "sparse_attn launch");
  return CSA2_OK;
}

}  // extern "C"
