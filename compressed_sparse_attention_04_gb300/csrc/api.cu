// Status strings, per-thread error messages and the device error word readers.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cmath>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace csa2 {

std::atomic<unsigned long long> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
RopeTurns rope_turns(float rope_base) {
  RopeTurns t;
  const long double two_pi = 6.283185307179586476925286766559005768L;
  for (int i = 0; i < 32; ++i) {
    const long double f = powl((long double)rope_base, -(long double)i / 32.0L) / two_pi;
    t.f[i] = (unsigned long long)llroundl(ldexpl(f, 64));   // f < 1/(2 pi): below 2^62
  }
  return t;
}
EncodeTiledFn tensor_map_encoder() {   // thread-safe static initialisation
  static const EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return EncodeTiledFn(nullptr);
  }();
  return fn;
}
bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("CSA2_NO_PDL");
    return !(v && v[0] == '1');
  }();
  return on;
}

namespace {
thread_local char g_msg[512] = "";
std::mutex g_mu;
std::vector<err_reader>& readers() {
  static std::vector<err_reader> v;
  return v;
}
}  // namespace

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(CSA2_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

void register_err_reader(err_reader f) {
  std::lock_guard<std::mutex> lk(g_mu);
  readers().push_back(f);
}

}  // namespace csa2

extern "C" {

const char* csa2_status_str(int s) {
  switch (s) {
    case CSA2_OK: return "CSA2_OK";
    case CSA2_ERR_INVALID_ARG: return "CSA2_ERR_INVALID_ARG";
    case CSA2_ERR_UNSUPPORTED: return "CSA2_ERR_UNSUPPORTED";
    case CSA2_ERR_WORKSPACE: return "CSA2_ERR_WORKSPACE";
    case CSA2_ERR_CUDA: return "CSA2_ERR_CUDA";
    case CSA2_ERR_TIMEOUT: return "CSA2_ERR_TIMEOUT";
    case CSA2_ERR_DEVICE_CHECK: return "CSA2_ERR_DEVICE_CHECK";
    default: return "CSA2_ERR_UNKNOWN";
  }
}

const char* csa2_last_error_message(void) { return csa2::g_msg; }

const char* csa2_version(void) { return "csa2-gb300 0.1 (sm_103a)"; }

unsigned long long csa2_kernel_launches(void) { return csa2::g_launches.load(); }

int csa2_last_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return csa2::cuda_fail(e, "cudaStreamSynchronize");
  unsigned word = 0;
  {
    std::lock_guard<std::mutex> lk(csa2::g_mu);
    for (auto f : csa2::readers()) word |= f();
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return csa2::cuda_fail(e, "reading device error word");
  if (word & csa2::ERR_TIMEOUT) return csa2::fail(CSA2_ERR_TIMEOUT, "a bounded device wait expired");
  if (word & csa2::ERR_BOUNDS)
    return csa2::fail(CSA2_ERR_DEVICE_CHECK, "a device-side bounds check fired");
  return CSA2_OK;
}

}  // extern "C"
