// Data movement around the expert GEMMs ("Scalable Pretraining of Large MoE
// LMs on Aurora Super Computer", §3.1, Algorithm 1):
//   permute  mlp_in = input[input_indices]           (stage 4)
//   combine  output reduction weighted by the gates  (stage 5, forward)
// Both run one warp per token and move rows as 16-byte vectors.  The permute
// reads each token row once and writes it to its k rows; the combine reads
// the k rows of a token and writes its output row once.  Rows are 2*d bytes
// of contiguous memory, so every access is coalesced on both sides.
//
// A row index outside [0, T*k) (the -1 the dispatch pass writes for a pair
// it could not place, or anything else a caller passes) is never used as an
// address: the permute skips that copy, the combine leaves that slot out of
// the sum, and the kernel records MOE_ERR_BAD_INDEX in `status` when one is
// given.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 16;  // one token per warp at 16k tokens: a single wave of warps
constexpr int kVecPerLane = 4;  // 16-byte vectors in flight per lane

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Row index of slot `lane` of token t, and whether every slot's row lies in
// [0, P) (lanes at or past k hold row 0).  A warp that meets a bad row
// records it once.
__device__ __forceinline__ int load_rows(const int32_t* __restrict__ dest_row, int64_t t, int k, int64_t P, int lane,
                                         unsigned& bad_slots, int32_t* status) {
  int r = (lane < k) ? __ldg(dest_row + t * k + lane) : 0;
  const bool bad = r < 0 || static_cast<int64_t>(r) >= P;
  bad_slots = __ballot_sync(0xffffffffu, bad);
  if (bad_slots != 0u && lane == 0) record_status(status, kStatusBadIndex);
  return r;
}

// One token's row to its k rows; kSkip as in combine_token.
template <bool kSkip>
__device__ __forceinline__ void permute_token(const uint4* __restrict__ x, int my_row, unsigned bad_slots, int64_t t,
                                              int k, int dvec, int lane, uint4* __restrict__ x_perm) {
  const uint4* src = x + t * dvec;
  for (int v0 = 0; v0 < dvec; v0 += 32 * kVecPerLane) {
    uint4 buf[kVecPerLane];
#pragma unroll
    for (int u = 0; u < kVecPerLane; ++u) {
      const int v = v0 + u * 32 + lane;
      if (v < dvec) buf[u] = ld_stream(src + v);
    }
    for (int j = 0; j < k; ++j) {
      const int64_t row = __shfl_sync(0xffffffffu, my_row, j);
      if (kSkip && ((bad_slots >> j) & 1u)) continue;  // warp-uniform
      uint4* dst = x_perm + row * dvec;
#pragma unroll
      for (int u = 0; u < kVecPerLane; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < dvec) dst[v] = buf[u];
      }
    }
  }
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
permute_kernel(const uint4* __restrict__ x, int64_t T, int dvec, const int32_t* __restrict__ dest_row, int k,
               uint4* __restrict__ x_perm, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t P = T * k;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5); t < T;
       t += warps_total) {
    unsigned bad_slots;
    const int my_row = load_rows(dest_row, t, k, P, lane, bad_slots, status);
    if (bad_slots == 0u)
      permute_token<false>(x, my_row, 0u, t, k, dvec, lane, x_perm);
    else
      permute_token<true>(x, my_row, bad_slots, t, k, dvec, lane, x_perm);
  }
}

__device__ __forceinline__ void accumulate_bf16x8(float (&acc)[8], const uint4& v, float w) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
  }
}

constexpr int kCombineVec = 2;

// One token's output row: its k rows weighted and summed in fp32 in slot
// order.  kSkip: some slot's row is out of range (bad_slots) and is left out
// of the sum; the usual case, every row valid, runs the loop without the
// per-slot test so that its loads pipeline across slots.
template <bool kSkip>
__device__ __forceinline__ void combine_token(const uint4* __restrict__ y, int my_row, float my_w, unsigned bad_slots,
                                              int64_t t, int k, int dvec, int lane, uint4* __restrict__ out) {
  for (int v0 = 0; v0 < dvec; v0 += 32 * kCombineVec) {
    float acc[kCombineVec][8];
#pragma unroll
    for (int u = 0; u < kCombineVec; ++u)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
    // slots in order j = 0..k-1: the fp32 sum has one fixed order
#pragma unroll 4
    for (int j = 0; j < k; ++j) {
      const int64_t row = __shfl_sync(0xffffffffu, my_row, j);
      const float wj = __shfl_sync(0xffffffffu, my_w, j);
      if (kSkip && ((bad_slots >> j) & 1u)) continue;  // warp-uniform
      const uint4* src = y + row * dvec;
#pragma unroll
      for (int u = 0; u < kCombineVec; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < dvec) accumulate_bf16x8(acc[u], ld_stream(src + v), wj);
      }
    }
#pragma unroll
    for (int u = 0; u < kCombineVec; ++u) {
      const int v = v0 + u * 32 + lane;
      if (v < dvec) {
        uint4 o;
        o.x = pack_bf16x2(acc[u][0], acc[u][1]);
        o.y = pack_bf16x2(acc[u][2], acc[u][3]);
        o.z = pack_bf16x2(acc[u][4], acc[u][5]);
        o.w = pack_bf16x2(acc[u][6], acc[u][7]);
        out[t * dvec + v] = o;
      }
    }
  }
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
combine_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ dest_row, const float* __restrict__ w,
               int64_t T, int k, int dvec, uint4* __restrict__ out, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t P = T * k;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5); t < T;
       t += warps_total) {
    unsigned bad_slots;
    const int my_row = load_rows(dest_row, t, k, P, lane, bad_slots, status);
    const float my_w = (w != nullptr && lane < k) ? __ldg(w + t * k + lane) : 1.0f;
    if (bad_slots == 0u)
      combine_token<false>(y, my_row, my_w, 0u, t, k, dvec, lane, out);
    else
      combine_token<true>(y, my_row, my_w, bad_slots, t, k, dvec, lane, out);
  }
}

int token_grid(int64_t T, int num_sms) {
  const int64_t want = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  return static_cast<int>(want < cap ? want : cap);
}

}  // namespace

cudaError_t launch_permute(const void* x, int64_t T, int d, const int32_t* dest_row, int k, void* x_perm,
                           int32_t* status, int num_sms, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  permute_kernel<<<token_grid(T, num_sms), kWarpsPerBlock * 32, 0, stream>>>(
      static_cast<const uint4*>(x), T, d / 8, dest_row, k, static_cast<uint4*>(x_perm), status);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* y, const int32_t* dest_row, const float* topk_w, int64_t T, int k, int d,
                           void* out, int32_t* status, int num_sms, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  combine_kernel<<<token_grid(T, num_sms), kWarpsPerBlock * 32, 0, stream>>>(
      static_cast<const uint4*>(y), dest_row, topk_w, T, k, d / 8, static_cast<uint4*>(out), status);
  return cudaGetLastError();
}

}  // namespace moe
