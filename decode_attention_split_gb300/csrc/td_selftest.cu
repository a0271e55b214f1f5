// td_selftest_wait_timeout: a diagnostic of the bounded wait every td kernel uses on its
// asynchronous copies. One CTA initialises an mbarrier that expects one arrival, never
// arrives on it and never issues a copy against it, then waits for its first phase with the
// kernels' wait (mbar_wait_bounded_for) and the caller's limit. The wait must give up, the
// kernel must set TD_DEV_WAIT_TIMEOUT in the caller's status word and return, and the
// device must stay usable. Nothing is in flight when the wait gives up.
#include "td_internal.h"
#include "td_device.cuh"

namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(long long limit, uint32_t *status, long long *waited) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    td::mbar_init(td::smem_u32(&bar), 1);
    td::fence_mbar_init();
  }
  __syncthreads();
  const long long t0 = clock64();
  const bool done = td::mbar_wait_bounded_for(td::smem_u32(&bar), 0u, limit);
  const long long t1 = clock64();
  // one decision for the CTA, as the kernels take it
  if (!__all_sync(0xffffffffu, done) && threadIdx.x == 0) {
    td::report(status, TD_DEV_WAIT_TIMEOUT);
    if (waited != nullptr) *waited = t1 - t0;
  }
}

}  // namespace

extern "C" td_status td_selftest_wait_timeout(long long limit_cycles, uint32_t *dev_status, long long *waited_cycles,
                                              void *stream) {
  if (dev_status == nullptr) return TD_ERR_INVALID_ARG;
  // at most about half a second at the GB300's clock: the wait always ends
  if (limit_cycles < 1 || limit_cycles > 1000000000LL) return TD_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dev_status) & 3u) != 0 || (reinterpret_cast<uintptr_t>(waited_cycles) & 7u) != 0)
    return TD_ERR_UNSUPPORTED;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_cycles, dev_status, waited_cycles);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TD_OK : td::cuda_fail(e);
}
