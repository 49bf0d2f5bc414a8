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

#include "common.cuh"

namespace {

// Scores of one call: B * Tq * row_len float32 values must fit.
constexpr size_t kScratchBytes = size_t(16) << 20;   // 16 MiB = 4 Mi scores
static __device__ __align__(256) unsigned char g_indexer_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_indexer_scratch on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return csa2::cuda_fail(e, "indexer_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return csa2::fail(CSA2_ERR_UNSUPPORTED, "indexer_noalloc: device ordinal %d not supported", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_indexer_scratch);
    if (e != cudaSuccess || !p)
      return csa2::cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                             "indexer_noalloc: cudaGetSymbolAddress of the scratch array");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
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
