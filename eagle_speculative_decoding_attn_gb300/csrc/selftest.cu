// tv_selftest_wait_timeout: the bounded-wait machinery every kernel of this
// library uses, made to expire on purpose.  One CTA waits on an mbarrier that
// nothing ever completes; the wait gives up after its time limit, the kernel
// records TV_DEV_TIMEOUT and returns, and the context stays usable.
#include "tv_common.cuh"

namespace tv {

__global__ void __launch_bounds__(64) wait_timeout_kernel(int32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_sh;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    abort_sh = 0;
  }
  __syncthreads();
  // no thread ever arrives: phase 0 never completes
  const bool ok = mbar_wait(&bar, 0, &abort_sh);
  if (!ok && threadIdx.x == 0) atomicOr(status, TV_DEV_TIMEOUT);
}

}  // namespace tv

extern "C" int tv_selftest_wait_timeout(int32_t* status, void* stream) {
  tv::clear_error();
  TV_REQUIRE(status, TV_ERR_INVALID_ARG, "tv_selftest_wait_timeout: NULL status");
  tv::wait_timeout_kernel<<<1, 64, 0, tv::as_stream(stream)>>>(status);
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}
