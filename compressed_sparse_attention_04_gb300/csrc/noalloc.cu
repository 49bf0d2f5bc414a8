// Indexer scores + top-k without any device allocation by the caller or the library.
//
// Some callers cannot hand the library a workspace: code that runs where allocating
// is not allowed or not possible (inside an allocator callback, in a process whose
// device memory is fully pre-reserved by another framework, or in a plain C host
// that has no allocator of its own wired to the GPU).  For them this file keeps the
// score scratch of csa2_indexer_score_topk in a fixed device array that is part of
// the library image itself: it comes into existence when the library's module is
// loaded on a device and stays until the process exits.
#include <mutex>

#include <cuda.h>

#include "common.cuh"

namespace {

// Scores of one call: B * Tq * row_len float32 values must fit.
constexpr size_t kScratchBytes = size_t(16) << 20;   // 16 MiB = 4 Mi scores
static __device__ __align__(256) unsigned char g_indexer_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// A __device__ array's address belongs to the CUDA context that loaded the module, not to
// the device: after cudaDeviceReset the primary context (and the array) is created anew,
// and a context made current through the driver API holds a copy of its own.  So each
// device slot remembers the context its address was looked up in, and a call made under
// another context looks the address up again.
struct ScratchSlot {
  CUcontext ctx;
  void* ptr;
};
ScratchSlot g_slot[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current_fn() {   // driver entry point, looked up once
  static const CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(p);
    return CtxGetCurrentFn(nullptr);
  }();
  return fn;
}

// Device address of g_indexer_scratch in the current context of the current device.
// With no context current yet (a thread's first runtime call), the symbol lookup itself
// makes the device's primary context current, so the context is read again after it.
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return csa2::cuda_fail(e, "indexer_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return csa2::fail(CSA2_ERR_UNSUPPORTED, "indexer_noalloc: device ordinal %d not supported", dev);
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (!get_ctx)
    return csa2::fail(CSA2_ERR_CUDA, "indexer_noalloc: driver entry point cuCtxGetCurrent not found");
  std::lock_guard<std::mutex> lk(g_mu);
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  ScratchSlot& slot = g_slot[dev];
  if (ctx == nullptr || slot.ptr == nullptr || slot.ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_indexer_scratch);
    if (e != cudaSuccess || !p)
      return csa2::cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                             "indexer_noalloc: cudaGetSymbolAddress of the scratch array");
    if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx)
      return csa2::fail(CSA2_ERR_CUDA, "indexer_noalloc: no current CUDA context");
    slot.ctx = ctx;
    slot.ptr = p;
  }
  *out = slot.ptr;
  return CSA2_OK;
}

}  // namespace

extern "C" {

size_t csa2_indexer_noalloc_max_scratch_bytes(void) { return kScratchBytes; }

int csa2_indexer_score_topk_noalloc(const void* q_idx, const float* w, int B, int Tq, int q_pos0,
                                    const uint8_t* codes, const uint8_t* scales, int n_cap,
                                    int n_entries, int m, const int32_t* cand, int nb, int blk,
                                    int k, int32_t* topk_out, float* blockmax_out,
                                    void* stream) {
  if (B <= 0 || Tq <= 0 || n_entries < 0 || (cand && (nb < 1 || blk < 1)))
    return csa2::fail(CSA2_ERR_INVALID_ARG, "indexer_noalloc: bad shape");
  const size_t need = csa2_indexer_workspace_size(B, Tq, n_entries, nb, blk, cand != nullptr);
  if (need > kScratchBytes)
    return csa2::fail(CSA2_ERR_UNSUPPORTED,
                      "indexer_noalloc: this call needs %zu bytes of score scratch but the "
                      "built-in array holds %zu; use csa2_indexer_score_topk with a workspace",
                      need, kScratchBytes);
  void* scratch = nullptr;
  int st = scratch_address(&scratch);
  if (st != CSA2_OK) return st;
  // Every score the top-k pass reads is written by the scoring pass of the same
  // call, so nothing in the array has to start at zero.
  return csa2_indexer_score_topk(q_idx, w, B, Tq, q_pos0, codes, scales, n_cap, n_entries, m,
                                 cand, nb, blk, k, topk_out, blockmax_out, nullptr, scratch,
                                 kScratchBytes, stream);
}

}  // extern "C"
