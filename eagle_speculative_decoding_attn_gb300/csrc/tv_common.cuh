// Shared host/device helpers of libtreeverify: status codes, argument checks,
// per-thread error text and device properties.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>
#include <cstdio>
#include <string>
#include "../../include/treeverify.h"
#include "tv_ptx.cuh"

namespace tv {

constexpr int kPageSize = 16;
constexpr int kMaxNodes = 64;

// ---------------------------------------------------------------- host errors
void set_error(const char* fmt, ...);
void clear_error();

#define TV_REQUIRE(cond, code, ...)      \
  do {                                   \
    if (!(cond)) {                       \
      ::tv::set_error(__VA_ARGS__);      \
      return (code);                     \
    }                                    \
  } while (0)

#define TV_CUDA_CHECK(expr)                                                        \
  do {                                                                             \
    cudaError_t _e = (expr);                                                       \
    if (_e != cudaSuccess) {                                                       \
      ::tv::set_error("%s failed: %s", #expr, cudaGetErrorString(_e));             \
      return TV_ERR_CUDA;                                                          \
    }                                                                              \
  } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count of the current device (cached per device id).
int current_sm_count();

// Unique id of the calling thread's current CUDA context (0: none yet).  The
// library keys what it caches per context on it, so that a device reset (which
// ends the context and loads the kernels again in a new one) is noticed.
cudaError_t current_context_id(unsigned long long* id);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (context, kernel).
cudaError_t ensure_smem_attr(const void* func, size_t bytes);
// A kernel that moves registers between its warpgroups (setmaxnreg) must have
// been built with exactly the per-thread count its split assumes: a smaller pool
// would leave an increase waiting forever.  cudaErrorInvalidKernelImage if not.
cudaError_t check_launch_regs(const void* func, int expected);

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Launch with programmatic dependent launch allowed: the kernel may be
// scheduled while the previous kernel on the stream is finishing.  Every kernel
// launched this way calls griddep_wait() before its first access to global
// memory, which returns once the previous kernel has completed and its writes
// are visible; a plain launch makes that call a no-op.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace tv
