// Checks of pieces every kernel shares.  The failure path: a bounded wait on
// an mbarrier phase that never completes gives up after its limit, records
// MOE_ERR_TIMEOUT in the workspace status word and returns, leaving the
// context usable (nothing here faults, traps or spins without a bound).  The
// activation functions: the exact device functions the expert-GEMM
// epilogues apply, elementwise, so that their error can be measured.  And a
// measurement tool: a kernel that holds a number of SMs for a bounded time,
// to see how the dynamically scheduled GEMMs share the rest.
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

__global__ void activation_kernel(const float* __restrict__ z, int64_t n, float* __restrict__ silu,
                                  float* __restrict__ sigmoid) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float v = z[i];
    silu[i] = silu_f32(v);
    sigmoid[i] = sigmoid_f32(v);
  }
}

// One block per SM it occupies: the block's dynamic shared memory (set by
// the launch) keeps any kernel that needs most of an SM's shared memory off
// that SM, and one thread sleeps until the block has existed for
// duration_ns.
__global__ void __launch_bounds__(32) occupy_kernel(uint64_t duration_ns) {
  extern __shared__ uint8_t hold[];
  if (threadIdx.x == 0) {
    hold[0] = 0;
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < duration_ns) __nanosleep(2000);
  }
}

}  // namespace

cudaError_t launch_occupy(int n_sms, uint64_t duration_ns, cudaStream_t stream) {
  if (n_sms == 0 || duration_ns == 0) return cudaSuccess;
  constexpr int kHold = 160 * 1024;  // over half of an SM's 228 KB: one block per SM
  cudaError_t err = cudaFuncSetAttribute(occupy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kHold);
  if (err != cudaSuccess) return err;
  occupy_kernel<<<n_sms, 32, kHold, stream>>>(duration_ns);
  return cudaGetLastError();
}

cudaError_t launch_activation(const float* z, int64_t n, float* silu, float* sigmoid, int num_sms,
                              cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int64_t want = (n + 255) / 256;
  const int grid = static_cast<int>(want < num_sms * 8 ? want : num_sms * 8);
  activation_kernel<<<grid, 256, 0, stream>>>(z, n, silu, sigmoid);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout(int32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 64, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
