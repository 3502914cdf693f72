// Check of the failure path shared by every kernel: a bounded wait on an
// mbarrier phase that never completes gives up after its limit, records
// MOE_ERR_TIMEOUT in the workspace status word and returns, leaving the
// context usable.  Nothing here faults, traps or spins without a bound.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// Warp 0 waits with the single-thread helper, warp 1 with the warp-wide
// one, both on a barrier that expects one arrival that never comes.
__global__ void __launch_bounds__(64) wait_timeout_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int never;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    never = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort_flag = &never;
  const int warp = threadIdx.x >> 5;
  if (warp == 0) {
    if ((threadIdx.x & 31) == 0 && !mbar_wait(&bar, 0, abort_flag, limit_ns)) record_status(status, kStatusTimeout);
  } else {
    if (!mbar_wait_warp(&bar, 0, abort_flag, limit_ns) && (threadIdx.x & 31) == 0)
      record_status(status, kStatusTimeout);
  }
}

}  // namespace

cudaError_t launch_wait_timeout(int32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 64, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
