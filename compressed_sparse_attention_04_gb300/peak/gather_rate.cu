// DRAM read rate of row gathers on this GPU: the denominator question for the attention kernel,
// which gathers the selected 1 KB cache rows.  Every SM runs one CTA that copies R rows of
// `row_bytes` into a shared-memory ring of four chunks with 16-byte cp.async (data never read),
// the chunk's row indices staged in shared memory first so that no copy waits on a load.
// Rows are either random over an 8 GB buffer or contiguous; 512 MB per launch after a 512 MB
// write that evicts the L2; best of three launches after one warm-up.
#include <cstdint>
#include <vector>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}

constexpr int T = 256, SLOTS = 4;

// chunk = cr rows; thread t copies piece t % P of rows t / P, t / P + T / P, ...
__global__ void __launch_bounds__(T, 1) gather_rows(const uint8_t* buf, const long long* idx, int R,
                                                    int cr, int row_bytes) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ long long sidx[SLOTS][192];   // rows per chunk: 48 KB / row_bytes <= 192
  const int tid = threadIdx.x, P = row_bytes / 16, rpp = T / P;
  const long long* my = idx + (long long)blockIdx.x * R;
  const uint32_t base = uint32_t(__cvta_generic_to_shared(sm));
  const int p = tid % P, r0 = tid / P;
  for (int c = 0; c < R / cr; ++c) {
    const int s = c % SLOTS;
    __syncthreads();   // every thread has issued the copies that read slot s's old indices
    for (int j = tid; j < cr; j += T) sidx[s][j] = __ldg(my + (long long)c * cr + j);
    __syncthreads();
    const uint32_t dst = base + uint32_t(s * cr * row_bytes);
    for (int r = r0; r < cr; r += rpp)
      cp16(dst + uint32_t(r * row_bytes + p * 16), buf + sidx[s][r] * row_bytes + p * 16);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group %0;" :: "n"(SLOTS - 1) : "memory");
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

}  // namespace

extern "C" {

// Read rate in GB/s of row gathers of `row_bytes` (256, 512, 1024, 2048 or 4096), random
// (random != 0) or contiguous rows, one 256-thread CTA per SM with 48 KB chunks.  Returns 0,
// or a CUDA error code.
int csa2peak_gather(int row_bytes, int random, double* gbs, double* ms_out) {
  if (row_bytes < 256 || row_bytes > 4096 || (row_bytes & (row_bytes - 1)) != 0) return int(cudaErrorInvalidValue);
  const size_t buf_bytes = 8ull << 30, per_launch = 512ull << 20, flush_bytes = 512ull << 20;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int cr = int(48 * 1024 / row_bytes);   // rows per chunk
  const size_t smem = size_t(SLOTS) * cr * row_bytes;
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gather_rows, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  uint8_t *buf = nullptr, *flush = nullptr;
  long long* idx = nullptr;
  const int R = sms > 0 ? int(per_launch / row_bytes / sms) / cr * cr : 0;
  if (e == cudaSuccess) e = cudaMalloc(&buf, buf_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&flush, flush_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&idx, size_t(sms) * R * sizeof(long long));
  if (e == cudaSuccess) e = cudaMemset(buf, 1, buf_bytes);
  if (e == cudaSuccess) {
    std::vector<long long> h(size_t(sms) * R);
    const unsigned long long n_rows = buf_bytes / row_bytes;
    unsigned long long x = 0x9E3779B97F4A7C15ull ^ unsigned(row_bytes);
    for (size_t i = 0; i < h.size(); ++i) {
      x ^= x << 13; x ^= x >> 7; x ^= x << 17;
      h[i] = random ? (long long)(x % n_rows) : (long long)i;
    }
    e = cudaMemcpy(idx, h.data(), h.size() * sizeof(long long), cudaMemcpyHostToDevice);
  }
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (e == cudaSuccess) e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  float best = 1e30f;
  for (int rep = 0; rep < 4 && e == cudaSuccess; ++rep) {   // rep 0 warms up
    e = cudaMemset(flush, rep, flush_bytes);
    if (e != cudaSuccess) break;
    cudaEventRecord(e0);
    gather_rows<<<sms, T, smem>>>(buf, idx, R, cr, row_bytes);
    cudaEventRecord(e1);
    e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaGetLastError();
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    if (rep > 0 && ms < best) best = ms;
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (idx) cudaFree(idx);
  if (flush) cudaFree(flush);
  if (buf) cudaFree(buf);
  if (e != cudaSuccess) return int(e);
  *ms_out = best;
  *gbs = double(sms) * R * row_bytes / (best * 1e-3) / 1e9;
  return 0;
}

}  // extern "C"
