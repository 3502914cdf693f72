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

// ---- the expert GEMMs' FP8 weight layout
//
// Codes of one projection, stored [E][K][N] (rows K = the GEMM's reduction
// index, columns N = its output features), go to 128-row tiles of 64 K
// values, one tile = 8 KB in the order (expert, tile, K block, row, k):
// gate/up tile t holds gate features 64t .. 64t+63 and the same up
// features, with row s = 32g + 16h + r for feature 64t + 16g + r of gate
// (h = 0) or up (h = 1); down tile t holds output features 128t + s.
constexpr int kCodeTile = 64;  // bytes of K per tile row, features per transpose block

__global__ void __launch_bounds__(256) pack_codes_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                                         int K, int C, int kind) {
  __shared__ uint8_t tile[kCodeTile][kCodeTile + 16];
  const int64_t e = blockIdx.z;
  const int c0 = blockIdx.x * kCodeTile, k0 = blockIdx.y * kCodeTile;
  const int t = threadIdx.x;
  // 64 K rows x 64 feature bytes in, 16 bytes per thread
  const uint8_t* s = src + (e * K + k0 + t / 4) * static_cast<int64_t>(C) + c0 + (t % 4) * 16;
  *reinterpret_cast<uint4*>(&tile[t / 4][(t % 4) * 16]) = __ldg(reinterpret_cast<const uint4*>(s));
  __syncthreads();
  // 64 feature rows of 64 K bytes out
  const int c = c0 + t / 4;
  int tile_i, row, ntiles;
  if (kind == 2) {  // down
    tile_i = c / 128;
    row = c % 128;
    ntiles = C / 128;
  } else {          // gate (0) or up (1)
    tile_i = c / 64;
    const int j = c % 64;
    row = (j / 16) * 32 + kind * 16 + j % 16;
    ntiles = C / 64;
  }
  const int kb = k0 / 64, nkb = K / 64;
  uint8_t v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = tile[(t % 4) * 16 + i][t / 4];
  uint8_t* d = dst + (((e * ntiles + tile_i) * nkb + kb) * 128 + row) * 64 + (t % 4) * 16;
  *reinterpret_cast<uint4*>(d) = *reinterpret_cast<const uint4*>(v);
}

// Scales of one projection (one fp32 per 128 consecutive stored values, so
// per (expert, K row, 128-feature block)) to one record per (expert,
// feature block, K block): gate/up 136 floats (64 gate scales, 4 zeros, 64 up
// scales, 4 zeros), down 64.  The scales are stored as they are.
__global__ void __launch_bounds__(256) pack_scales_kernel(const float* __restrict__ gate_or_down,
                                                          const float* __restrict__ up, float* __restrict__ dst,
                                                          int E, int K, int C, int gate_up) {
  const int nfb = C / 128, nkb = K / 64, rec = gate_up ? kFp8GateUpRecord : kFp8DownRecord;
  const int64_t total = static_cast<int64_t>(E) * nfb * nkb * rec;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(i % rec);
    const int64_t r = i / rec;
    const int kb = static_cast<int>(r % nkb);
    const int fb = static_cast<int>((r / nkb) % nfb);
    const int64_t e = r / (static_cast<int64_t>(nkb) * nfb);
    float v = 0.0f;
    const float* src = gate_or_down;
    int kk = j;
    if (gate_up && j >= 68) {
      src = up;
      kk = j - 68;
    }
    if (kk < 64) v = __ldg(src + (e * K + kb * 64 + kk) * nfb + fb);
    dst[i] = v;
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

size_t fp8_packed_bytes(int E, int d, int f, size_t* offsets) {
  const size_t edf = static_cast<size_t>(E) * d * f;
  const size_t sc_gu = align_up(static_cast<size_t>(E) * (f / 128) * (d / 64) * kFp8GateUpRecord * 4);
  const size_t sc_dn = align_up(static_cast<size_t>(E) * (d / 128) * (f / 64) * kFp8DownRecord * 4);
  if (offsets) {
    offsets[0] = 0;             // gate/up codes
    offsets[1] = 2 * edf;       // down codes
    offsets[2] = 3 * edf;       // gate/up scale records
    offsets[3] = 3 * edf + sc_gu;  // down scale records
  }
  return 3 * edf + sc_gu + sc_dn;
}

cudaError_t launch_pack_weights_fp8(const uint8_t* gate_codes, const float* gate_scales, const uint8_t* up_codes,
                                    const float* up_scales, const uint8_t* down_codes, const float* down_scales,
                                    int E, int d, int f, void* packed, int num_sms, cudaStream_t stream) {
  size_t off[4];
  fp8_packed_bytes(E, d, f, off);
  auto* base = static_cast<uint8_t*>(packed);
  // gate and up: stored [E][d][f] (K = d, features f); down: [E][f][d] (K = f, features d)
  const dim3 g_gu(f / kCodeTile, d / kCodeTile, E), g_dn(d / kCodeTile, f / kCodeTile, E);
  pack_codes_kernel<<<g_gu, 256, 0, stream>>>(gate_codes, base + off[0], d, f, 0);
  pack_codes_kernel<<<g_gu, 256, 0, stream>>>(up_codes, base + off[0], d, f, 1);
  pack_codes_kernel<<<g_dn, 256, 0, stream>>>(down_codes, base + off[1], f, d, 2);
  pack_scales_kernel<<<num_sms * 4, 256, 0, stream>>>(gate_scales, up_scales, reinterpret_cast<float*>(base + off[2]),
                                                     E, d, f, 1);
  pack_scales_kernel<<<num_sms * 4, 256, 0, stream>>>(down_scales, nullptr, reinterpret_cast<float*>(base + off[3]),
                                                     E, f, d, 0);
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
