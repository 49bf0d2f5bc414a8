// Dense FP4 tensor-core throughput of this GPU: the denominator of the prefill scorer's
// tensor-pipe fraction.  Every SM runs one CTA whose single issuing thread streams
// block-scaled FP4 MMAs (kind::mxf4nvf4, scale_vec::4X: E2M1 operands, E4M3 scales per 16
// elements, float32 accumulate) of shape M x N x 64 from shared memory into TMEM, back to
// back, then waits for them.  Operands and scales are zero: the rate does not depend on the
// values.  FLOPs = 2 M N 64 per MMA; TFLOP/s = all SMs' FLOPs / the launch's event time.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// K-major operand without swizzle: 8-row x 16-byte core matrices, 128 B apart along K,
// 8-row groups 512 B apart (rows of 64 FP4 elements = 32 bytes)
__device__ __forceinline__ uint64_t desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t(128u >> 4) << 16;
  d |= uint64_t(512u >> 4) << 32;
  d |= uint64_t(1) << 46;
  return d;
}

constexpr int T = 128;
constexpr uint32_t SMEM = 48 * 1024;   // A (128 x 32 B) + B (256 x 32 B), with room

__global__ void __launch_bounds__(T, 1) mxf4_stream(int M, int N, int iters, unsigned* err) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t tslot;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < int(SMEM / 16); i += T) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" :: "r"(smem_u32(&tslot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(smem_u32(&done)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tslot;
  // scale factors: zero words in TMEM columns 256.. (A) and 272.. (B)
  {
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1};"
                 :: "r"(tmem + lane_base + 256), "r"(0u) : "memory");
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1};"
                 :: "r"(tmem + lane_base + 272), "r"(0u) : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (tid == 0) {
    const uint32_t idesc = (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
    const uint64_t da = desc(smem_u32(sm)), db = desc(smem_u32(sm + 16 * 1024));
    for (int i = 0; i < iters; ++i) {
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
          "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
          :: "r"(tmem), "l"(da), "l"(db), "r"(idesc), "r"(tmem + 256), "r"(tmem + 272), "r"(uint32_t(i > 0)));
    }
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(&done)) : "memory");
    uint32_t ok = 0;
    for (uint32_t it = 0; it < (1u << 26) && !ok; ++it)
      asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                   : "=r"(ok) : "r"(smem_u32(&done)) : "memory");
    if (!ok) atomicOr(err, 1u);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" :: "r"(tmem));
}

}  // namespace

extern "C" {

// Dense block-scaled FP4 rate with MMAs of M x N x 64 (M = 128; N a multiple of 16 up to
// 256), `iters` per SM, on the current device.  Writes the achieved TFLOP/s and the launch
// time; returns 0, or a nonzero CUDA error / 1000 when a wait expired.
int csa2peak_mxf4(int M, int N, int iters, double* tflops, double* ms_out) {
  if (M != 128 || N < 16 || N > 256 || N % 16 != 0 || iters < 1) return int(cudaErrorInvalidValue);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(mxf4_stream, cudaFuncAttributeMaxDynamicSharedMemorySize, int(SMEM));
  unsigned* err = nullptr;
  if (e == cudaSuccess) e = cudaMalloc(&err, sizeof(unsigned));
  if (e == cudaSuccess) e = cudaMemset(err, 0, sizeof(unsigned));
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (e == cudaSuccess) e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  float best = 1e30f;
  for (int rep = 0; rep < 4 && e == cudaSuccess; ++rep) {   // rep 0 warms up
    cudaEventRecord(e0);
    mxf4_stream<<<sms, T, SMEM>>>(M, N, iters, err);
    cudaEventRecord(e1);
    e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaGetLastError();
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    if (rep > 0 && ms < best) best = ms;
  }
  unsigned herr = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&herr, err, sizeof(unsigned), cudaMemcpyDeviceToHost);
  if (err) cudaFree(err);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (e != cudaSuccess) return int(e);
  if (herr) return 1000;
  *ms_out = best;
  *tflops = 2.0 * M * N * 64.0 * double(iters) * sms / (best * 1e-3) / 1e12;
  return 0;
}

}  // extern "C"
