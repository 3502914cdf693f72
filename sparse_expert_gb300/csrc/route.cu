// Stage 1 of the layer: Softmax and TopK of the router logits, one warp per
// token ("Scalable Pretraining of Large MoE LMs on Aurora Super Computer",
// §3.1, Algorithm 1, stage 1).  Optionally adds each selection to a
// per-expert histogram (the token counts of stage 2) so that the index pass
// can start from complete counts without another read of the indices.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;  // tokens per block

// Strict total order of (value, expert): larger value first, then the
// smaller expert index.  -0.0 == +0.0 under IEEE comparison.
__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
  return v > bv || (v == bv && e < be);
}

// NV logits per lane: lane l holds experts l, l+32, ..., l+32*(NV-1).
template <int NV>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_topk_kernel(const float* __restrict__ logits, int64_t T, int E, int k, int renormalize,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ counts) {
  extern __shared__ int32_t s_hist[];  // [E] when counts != nullptr
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (counts) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
    __syncthreads();
  }

  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * kRouteWarps;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kRouteWarps + warp; t < T; t += warps_total) {
    const float* row = logits + t * E;
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? __ldg(row + e) : -INFINITY;
    }
    // the maximum is the best expert's logit; find it first for the softmax
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < NV; ++i) mx = fmaxf(mx, v[i]);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    float denom_all = 0.f;
    if (!renormalize) {
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (lane + 32 * i < E) denom_all += expf(v[i] - mx);
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) denom_all += __shfl_xor_sync(0xffffffffu, denom_all, s);
    }

    // k rounds of a warp argmax under the total order; the winner is removed
    float my_val = 0.f;  // lane j keeps the j-th selection
    int my_idx = 0;
    uint32_t taken = 0;  // bit i: this lane's expert lane + 32*i is already selected
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && better(v[i], e, bv, be)) {
          bv = v[i];
          be = e;
        }
      }
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, s);
        const int oe = __shfl_xor_sync(0xffffffffu, be, s);
        if (better(ov, oe, bv, be)) {
          bv = ov;
          be = oe;
        }
      }
      if (lane == j) {
        my_val = bv;
        my_idx = be;
      }
      // remove the winner (it lives in lane be % 32, slot be / 32)
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (lane + 32 * i == be) taken |= 1u << i;
    }
    // gates
    const float z = (lane < k) ? expf(my_val - mx) : 0.f;
    float denom = denom_all;
    if (renormalize) {
      denom = z;
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, s);
    }
    if (lane < k) {
      topk_idx[t * k + lane] = my_idx;
      topk_w[t * k + lane] = z / denom;
      if (counts) atomicAdd(&s_hist[my_idx], 1);
    }
  }

  if (counts) {
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      const int c = s_hist[e];
      if (c) atomicAdd(&counts[e], c);
    }
  }
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, int64_t T, int E, int k, int renormalize, int32_t* topk_idx,
                              float* topk_w, int32_t* counts, int num_sms, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int64_t blocks_needed = (T + kRouteWarps - 1) / kRouteWarps;
  const int64_t max_blocks = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(blocks_needed < max_blocks ? blocks_needed : max_blocks);
  const size_t smem = counts ? static_cast<size_t>(E) * sizeof(int32_t) : 0;
  const int nv = (E + 31) / 32;
#define MOE_ROUTE_CASE(NV)                                                                                     \
  route_topk_kernel<NV><<<grid, kRouteWarps * 32, smem, stream>>>(logits, T, E, k, renormalize, topk_idx, topk_w, \
                                                                  counts);                                     \
  break;
  switch (nv <= 1 ? 1 : nv <= 2 ? 2 : nv <= 4 ? 4 : nv <= 8 ? 8 : nv <= 12 ? 12 : nv <= 16 ? 16 : 32) {
    case 1: MOE_ROUTE_CASE(1)
    case 2: MOE_ROUTE_CASE(2)
    case 4: MOE_ROUTE_CASE(4)
    case 8: MOE_ROUTE_CASE(8)
    case 12: MOE_ROUTE_CASE(12)
    case 16: MOE_ROUTE_CASE(16)
    default: MOE_ROUTE_CASE(32)
  }
#undef MOE_ROUTE_CASE
  return cudaGetLastError();
}

}  // namespace moe
