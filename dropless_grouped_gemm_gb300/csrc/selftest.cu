// selftest.cu - exercises the bounded wait every kernel of the library uses
// (ptx.cuh: mbar_wait_for), without faulting or hanging the GPU.
//
// One warp initialises two mbarriers in shared memory.  The first is
// completed by an arrival, so waiting on it must succeed at once.  Nothing
// ever arrives on the second, so the wait must give up after `limit_ns`,
// raise the abort flag and report MOE_DEV_TIMEOUT, exactly as a stalled
// pipeline role would.  Nothing asynchronous (TMA, MMA) is in flight.
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace moe {
namespace {

__global__ void bounded_wait_selftest(uint64_t limit_ns, int32_t* err, int32_t* waited_us) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive(&bars[0]);                               // completes phase 0 of bars[0]
    volatile int* ab = &abort_flag;
    const bool ok0 = mbar_wait_for(&bars[0], 0, ab, limit_ns);
    const uint64_t t0 = globaltimer_ns();
    const bool ok1 = mbar_wait_for(&bars[1], 0, ab, limit_ns);   // never completes
    const uint64_t t1 = globaltimer_ns();
    *waited_us = static_cast<int32_t>((t1 - t0) / 1000u);
    if (!ok0) set_err(err, 16);                          // must not happen
    if (!ok1 && *ab) set_err(err, MOE_DEV_TIMEOUT);
  }
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int limit_us, int32_t* err, int32_t* waited_us,
                                         cudaStream_t s) {
  bounded_wait_selftest<<<1, 32, 0, s>>>(static_cast<uint64_t>(limit_us) * 1000u, err, waited_us);
  return cudaGetLastError();
}

}  // namespace moe
