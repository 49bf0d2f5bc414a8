// Device twin of synth/philox.py: the same Philox4x32-10 words and the same
// float32 operations, so every element equals the host generator's bit for bit.
// Generator: Salmon et al., "Parallel random numbers: as easy as 1, 2, 3" (SC'11).
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace {

struct U4 { uint32_t a, b, c, d; };

__device__ __forceinline__ U4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                             uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    k0 += 0x9E3779B9u; k1 += 0xBB67AE85u;
  }
  return {c0, c1, c2, c3};
}

__device__ __forceinline__ float ih_normal(uint64_t i, uint32_t seed, uint32_t stream,
                                           float sigma) {
  const U4 r = philox4x32_10(uint32_t(i), uint32_t(i >> 32), 0u, 0u, seed, stream);
  int32_t acc = int32_t(2u * (r.a >> 10) + 1u) + int32_t(2u * (r.b >> 10) + 1u) +
                int32_t(2u * (r.c >> 10) + 1u) + int32_t(2u * (r.d >> 10) + 1u) -
                (1 << 24);
  // same constant as the host: float32(sqrt(3) / 2^23)
  const float kScale = __uint_as_float(0x345db3d7u);  // 0x1.bb67aep-23
  const float z = __fmul_rn(float(acc), kScale);
  return __fmul_rn(z, sigma);
}

__global__ void k_normal_bf16(__nv_bfloat16* out, uint64_t n, uint64_t start, uint32_t seed,
                              uint32_t stream, float sigma) {
  for (uint64_t j = blockIdx.x * uint64_t(blockDim.x) + threadIdx.x; j < n;
       j += uint64_t(gridDim.x) * blockDim.x)
    out[j] = __float2bfloat16_rn(ih_normal(start + j, seed, stream, sigma));
}

__global__ void k_normal_f32(float* out, uint64_t n, uint64_t start, uint32_t seed,
                             uint32_t stream, float sigma) {
  for (uint64_t j = blockIdx.x * uint64_t(blockDim.x) + threadIdx.x; j < n;
       j += uint64_t(gridDim.x) * blockDim.x)
    out[j] = ih_normal(start + j, seed, stream, sigma);
}

__global__ void k_u32(uint32_t* out, uint64_t n, uint64_t start, uint32_t seed,
                      uint32_t stream) {
  for (uint64_t j = blockIdx.x * uint64_t(blockDim.x) + threadIdx.x; j < n;
       j += uint64_t(gridDim.x) * blockDim.x) {
    const uint64_t i = start + j;
    out[j] = philox4x32_10(uint32_t(i), uint32_t(i >> 32), 0u, 0u, seed, stream).a;
  }
}

unsigned grid_for(uint64_t n) {
  uint64_t g = (n + 255) / 256;
  if (g > 152ull * 64) g = 152ull * 64;
  return unsigned(g < 1 ? 1 : g);
}

}  // namespace

extern "C" {

// All three fill n elements of `out` (device memory) with elements start..start+n-1
// of the given (seed, stream).  Return 0 or the cudaError_t of the launch.
int synth_normal_bf16(void* out, uint64_t n, uint64_t start, uint32_t seed, uint32_t stream,
                      float sigma, void* cuda_stream) {
  if (n == 0) return 0;
  k_normal_bf16<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(
      (__nv_bfloat16*)out, n, start, seed, stream, sigma);
  return int(cudaGetLastError());
}

int synth_normal_f32(void* out, uint64_t n, uint64_t start, uint32_t seed, uint32_t stream,
                     float sigma, void* cuda_stream) {
  if (n == 0) return 0;
  k_normal_f32<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(
      (float*)out, n, start, seed, stream, sigma);
  return int(cudaGetLastError());
}

int synth_u32(void* out, uint64_t n, uint64_t start, uint32_t seed, uint32_t stream,
              void* cuda_stream) {
  if (n == 0) return 0;
  k_u32<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>((uint32_t*)out, n, start, seed,
                                                            stream);
  return int(cudaGetLastError());
}

}  // extern "C"
