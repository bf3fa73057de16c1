// Host-side helpers shared by every entry point: thread-local error text,
// version string, cached device properties.
#include <cstdarg>
#include <cudaTypedefs.h>
#include <map>
#include <mutex>
#include <utility>
#include "tv_common.cuh"

namespace tv {

static thread_local std::string g_last_error;

void set_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
}

void clear_error() { g_last_error.clear(); }

int current_sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

cudaError_t current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_ctx = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_ctx = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  *id = 0;
  if (!get_ctx || !get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
  if (ctx == nullptr) return cudaSuccess;
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

cudaError_t ensure_smem_attr(const void* func, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<unsigned long long, const void*>, size_t> done;
  unsigned long long ctx = 0;
  cudaError_t e = current_context_id(&ctx);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (ctx != 0) {
    auto it = done.find(std::make_pair(ctx, func));
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
  }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  if (ctx == 0 && current_context_id(&ctx) != cudaSuccess) return cudaSuccess;  // not cached: set again next time
  if (ctx != 0) done[std::make_pair(ctx, func)] = bytes;
  return cudaSuccess;
}

cudaError_t check_launch_regs(const void* func, int expected) {
  static std::mutex mu;
  static std::map<const void*, int> regs;
  std::lock_guard<std::mutex> lock(mu);
  auto it = regs.find(func);
  if (it == regs.end()) {
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, func);
    if (e != cudaSuccess) return e;
    it = regs.emplace(func, fa.numRegs).first;
  }
  return it->second == expected ? cudaSuccess : cudaErrorInvalidKernelImage;
}

}  // namespace tv

extern "C" const char* tv_last_error(void) { return tv::g_last_error.c_str(); }

extern "C" const char* tv_version(void) { return "treeverify 0.1 (sm_103a)"; }
