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
// attn_simt_kernel: one CTA per (query row, group of 8 heads), one warp per head.
// Rows of A (top-k slots then window rows) stream through shared memory in tiles of
// 32; lane j scores row j of the tile; an online softmax keeps (max, sum) per head
// and every lane accumulates 16 of the 512 output dims.
#include "common.cuh"

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

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" {

size_t csa2_sparse_attn_workspace_size(int B, int Tq, int H, int k, int window) {
  (void)B; (void)Tq; (void)H; (void)k; (void)window;
  return 0;
}

int csa2_sparse_attn(const void* q, int B, int Tq, int H, int q_pos0, const void* kv_cache,
                     int n_cap, int n_entries, const int32_t* topk, int k, const void* swa_kv,
                     int S, int swa_pos0, int window, const float* sink, float scale, void* out,
                     float* lse_out, void* workspace, size_t ws_bytes, void* stream) {
  (void)workspace; (void)ws_bytes;
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
  attn_simt_kernel<<<unsigned(rows * n_hg), AT_T, 0, (cudaStream_t)stream>>>(aa);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "sparse_attn launch");
  return CSA2_OK;
}

}  // extern "C"
