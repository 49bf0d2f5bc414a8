// Shared device/host helpers of libcsa2 (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <cstddef>
#include <cmath>

#include "../../include/csa2.h"

namespace csa2 {

// ------------------------------------------------------------------ host side
// Records a one-line reason for the calling thread and returns `status`.
int fail(int status, const char* fmt, ...);
// Counts one kernel launch (csa2_kernel_launches reads the total).
void note_launch();
// Records a timing event on `stream`; inside a stream capture it becomes an event-record
// node of the graph (a plain record there would only mark a dependency).
inline void record_stage_event(cudaEvent_t e, cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(stream, &cs);
  if (cs == cudaStreamCaptureStatusActive) cudaEventRecordWithFlags(e, stream, cudaEventRecordExternal);
  else cudaEventRecord(e, stream);
}
int cuda_fail(cudaError_t e, const char* what);

// Programmatic dependent launch.  A kernel started by launch_k() may begin while the kernel
// before it on the stream is finishing: its launch then overlaps that kernel's last CTAs.
// Before pdl_wait() it may touch nothing but its own shared memory: pdl_wait() returns once
// the previous kernel has completed and its writes are visible.  Kernels do not trigger their
// successor early (griddepcontrol.launch_dependents): successor CTAs placed beside a running
// kernel and waiting for it slowed it down (measured: a 64-row top-k 11 -> 20 us), so each
// kernel's successor is released as its CTAs exit.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Whether launches carry the programmatic-serialization attribute (default on; the
// environment variable CSA2_NO_PDL=1 turns it off).
bool pdl_enabled();

// Launch `kernel` on `st` with programmatic serialization and, when cluster_x > 1, a
// cluster of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// launch_k() with a 1-CTA cluster shape, returning cuda_fail(error, where) on failure.
#define CSA2_LAUNCH(where, kernel, grid, block, smem, stream, ...)                              \
  do {                                                                                        \
    const cudaError_t le_ = ::csa2::launch_k(kernel, dim3(grid), dim3(block), size_t(smem),   \
                                             (cudaStream_t)(stream), 1u, __VA_ARGS__);        \
    if (le_ != cudaSuccess) return ::csa2::cuda_fail(le_, where);                             \
  } while (0)

// cuTensorMapEncodeTiled from the driver, looked up once (null when unavailable).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Device error word bits (OR-ed by kernels, read by csa2_last_device_status).
enum : unsigned { ERR_BOUNDS = 1u, ERR_TIMEOUT = 2u };

// Each translation unit that reports device errors owns one word and registers a
// reader; csa2_last_device_status ORs all of them.
using err_reader = unsigned (*)();
void register_err_reader(err_reader f);

// csa2_indexer_score_topk with two optional events recorded between the scoring
// launch and the top-k launch (used by the runner's per-stage timing), and the
// tensor-core decode scorer's wait bound and stall switch (csa2_indexer_score_topk_bounded).
int indexer_impl(const void* q_idx, const float* w, int B, int Tq, int q_pos0,
                 const uint8_t* codes, const uint8_t* scales, int n_cap, int n_entries, int m,
                 const int32_t* cand, int nb, int blk, int k, int32_t* topk_out,
                 float* blockmax_out, float* scores_out, void* workspace, size_t ws_bytes,
                 void* stream, cudaEvent_t ev_score_end, cudaEvent_t ev_topk_begin,
                 unsigned wait_limit = 0, int stall = 0, int* used_bounded = nullptr);

// The compressor (csa2_compress, or csa2_compress_chunk when state is given) whose epilogue
// also writes the new entries' indexer keys (as csa2_index_k_quant would, bit for bit) when
// the call has few entries; *fused tells whether it did -- if not, the caller runs
// csa2_index_k_quant on kv_pre.
int compress_index_k(const void* x, int B, int T, int hidden, int m, int pos0, const void* w_kv,
                     const void* w_gate, const float* norm_w, float eps, float rope_base,
                     float* state, void* kv_cache, int n_cap, float* kv_pre, void* workspace,
                     size_t ws_bytes, const void* w_ik, uint8_t* idx_codes, uint8_t* idx_scales,
                     void* stream, bool* fused);

// Entry positions visible to query position t (entry s covers tokens s*m..s*m+m-1).
__host__ __device__ inline int n_visible(long long t, int m, int n_entries) {
  long long v = (t + 1) / m;
  if (v < 0) v = 0;
  return int(v < n_entries ? v : n_entries);
}

// ------------------------------------------------------------------ device side
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(uint32_t(b) << 16);
}

// Order-preserving map float -> uint32 (larger float -> larger key); -0 == +0.
__device__ __forceinline__ uint32_t f32_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// E2M1 magnitude of code & 7 (0, .5, 1, 1.5, 2, 3, 4, 6): exponent e = c >> 1, mantissa
// bit c & 1; e == 0 is the subnormal 0.5 * m, otherwise 2^(e-1) * (1 + m/2).
__device__ __forceinline__ float e2m1_mag(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  return e == 0 ? 0.5f * float(m) : __uint_as_float(((e + 126u) << 23) | (m << 22));
}

__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const float v = e2m1_mag(c);
  return (c & 8u) ? -v : v;
}

// E4M3 (OCP FN) byte -> float: bias 7, subnormals m * 2^-9.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  float v = (e == 0) ? float(m) * 0.001953125f
                     : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (b & 0x80u) ? -v : v;
}

// float32 >= 0 -> E4M3 byte, round to nearest even, saturating at 448.
// Subnormal range (x < 2^-6): m * 2^-9 with m = rint(x * 512).  Normal range: round
// the 23-bit mantissa to 3 bits (a carry moves into the exponent), re-bias 127 -> 7.
__device__ __forceinline__ uint32_t e4m3_rne_satfinite(float x) {
  if (!(x < 448.0f)) return 0x7Eu;
  if (x < 0.015625f) return uint32_t(rintf(x * 512.0f));
  const uint32_t b = __float_as_uint(x);
  uint32_t q = b >> 20;
  const uint32_t rem = b & 0xFFFFFu;
  if (rem > 0x80000u || (rem == 0x80000u && (q & 1u))) ++q;
  const uint32_t code = q - (120u << 3);
  return code > 0x7Eu ? 0x7Eu : code;
}

// |u| -> E2M1 magnitude code, nearest with ties to the even code, saturating at 6.
__device__ __forceinline__ uint32_t e2m1_rne_mag(float a) {
  if (a <= 0.25f) return 0u;
  if (a < 0.75f) return 1u;
  if (a <= 1.25f) return 2u;
  if (a < 1.75f) return 3u;
  if (a <= 2.5f) return 4u;
  if (a < 3.5f) return 5u;
  if (a <= 5.0f) return 6u;
  return 7u;
}

// One 32-value block held one value per lane of a full warp: returns this lane's
// 4-bit code and (same on all lanes) the E4M3 scale byte.
__device__ __forceinline__ uint32_t fp4_quant_lane(float v, uint32_t& scale_byte) {
  float a = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const uint32_t sb = e4m3_rne_satfinite(__fdiv_rn(a, 6.0f));
  scale_byte = sb;
  if (sb == 0u) return 0u;
  const float s = e4m3_value(sb);
  const float u = __fdiv_rn(v, s);
  const uint32_t sign = (__float_as_uint(u) >> 31) << 3;
  return sign | e2m1_rne_mag(fabsf(u));
}

// FP8 window-KV group scale: the smallest k >= -126 with amax <= 448 * 2^k.  With amax =
// 1.m * 2^(E-127) and 448 = 1.75 * 2^8: k = E - 135, plus one when 1.m > 1.75 (mantissa
// field above 0x600000); zero and subnormal amax give -126.
__device__ __forceinline__ int fp8_scale_exp(float amax) {
  const uint32_t bits = __float_as_uint(amax), E = bits >> 23, mant = bits & 0x7FFFFFu;
  const int k = E == 0 ? -126 : int(E) - 135 + (mant > 0x600000u ? 1 : 0);
  return k < -126 ? -126 : k;
}

// RoPE angles.  Pair i (of 32) of the last 64 dims turns by pos * theta_i, theta_i =
// base^(-i/32).  t.f[i] holds theta_i / (2 pi) as a 64-bit binary fraction (computed on the
// host in extended precision), so the wrapping 64-bit product pos * t.f[i] is the angle's
// fractional turn; read as a signed fraction in [-1/2, 1/2) turn it goes to float for sincospif.
// Angle error about 2e-7 rad for any position below 2^40; no double-precision arithmetic.
struct RopeTurns {
  unsigned long long f[32];
};
RopeTurns rope_turns(float rope_base);

__device__ __forceinline__ void rope_cs(long long pos, int i, const RopeTurns& t, float& c, float& s) {
  const unsigned long long x = (unsigned long long)pos * t.f[i];
  const float turns = __ll2float_rn((long long)x) * 5.42101086242752217e-20f;   // 2^-64
  sincospif(2.0f * turns, &s, &c);
}

}  // namespace csa2

// Defines a translation-unit-local device error word `name` plus a reader that
// returns and clears it, registered with csa2_last_device_status.
#define CSA2_DEFINE_ERR_WORD(name)                                                  \
  static __device__ unsigned name;                                                  \
  static unsigned name##_read() {                                                   \
    unsigned v = 0, z = 0;                                                          \
    if (cudaMemcpyFromSymbol(&v, name, sizeof(v)) != cudaSuccess) return 0;         \
    cudaMemcpyToSymbol(name, &z, sizeof(z));                                        \
    return v;                                                                       \
  }                                                                                 \
  static const int name##_registered = (csa2::register_err_reader(&name##_read), 0);
