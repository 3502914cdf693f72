// Blockwise FP8 (E4M3) weights ("Training a 1T-Params MoE on EU public
// infrastructure", FP8 expert weight all-gather): blocks of 128 consecutive
// values, each scaled into the E4M3 range by one fp32 scale and cast; the
// receiver dequantises to bf16 before the expert computation.
//   scale = amax / 448 (1 for an all-zero block), code = E4M3(w / scale)
//   with fp32 division and round-to-nearest-even, saturating at +-448;
//   dequantised w' = bf16(E4M3 value * scale), the product in fp32.
// One warp per block for the encoding (each lane holds 4 values), one
// thread per 4 values for the decoding.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kBlock = 128;
constexpr float kE4M3Max = 448.0f;

__global__ void __launch_bounds__(256) quantize_kernel(const __nv_bfloat16* __restrict__ w, int64_t nblocks,
                                                       uint32_t* __restrict__ codes, float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); b < nblocks;
       b += warps) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(w + b * kBlock) + lane);
    const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    const float v[4] = {__low2float(p0), __high2float(p0), __low2float(p1), __high2float(p1)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, s));
    const float scale = amax > 0.0f ? amax / kE4M3Max : 1.0f;
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(v[i] / scale, __NV_SATFINITE, __NV_E4M3);
      packed |= static_cast<uint32_t>(c) << (8 * i);
    }
    codes[b * (kBlock / 4) + lane] = packed;
    if (lane == 0) scales[b] = scale;
  }
}

__global__ void __launch_bounds__(256) dequantize_kernel(const uint32_t* __restrict__ codes,
                                                         const float* __restrict__ scales, int64_t nquads,
                                                         uint2* __restrict__ out) {
  for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < nquads;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t c = __ldg(codes + q);
    const float scale = __ldg(scales + q / (kBlock / 4));
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>((c >> (8 * i)) & 0xFF), __NV_E4M3);
      v[i] = __half2float(__half(h)) * scale;
    }
    uint2 o;
    o.x = pack_bf16x2(v[0], v[1]);
    o.y = pack_bf16x2(v[2], v[3]);
    out[q] = o;
  }
}

int grid_for(int64_t items, int per_block, int num_sms) {
  const int64_t want = (items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(num_sms) * 16;
  return static_cast<int>(want < cap ? want : cap);
}

}  // namespace

cudaError_t launch_quantize_fp8(const void* w, int64_t n, uint8_t* codes, float* scales, int num_sms,
                                cudaStream_t stream) {
  const int64_t nblocks = n / kBlock;
  if (nblocks == 0) return cudaSuccess;
  quantize_kernel<<<grid_for(nblocks, 8, num_sms), 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(w), nblocks,
                                                                     reinterpret_cast<uint32_t*>(codes), scales);
  return cudaGetLastError();
}

cudaError_t launch_dequantize_fp8(const uint8_t* codes, const float* scales, int64_t n, void* out, int num_sms,
                                  cudaStream_t stream) {
  const int64_t nquads = n / 4;
  if (nquads == 0) return cudaSuccess;
  dequantize_kernel<<<grid_for(nquads, 256, num_sms), 256, 0, stream>>>(reinterpret_cast<const uint32_t*>(codes),
                                                                        scales, nquads, static_cast<uint2*>(out));
  return cudaGetLastError();
}

}  // namespace moe
