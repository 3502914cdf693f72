// One-time layout transform of the expert weights for the grouped GEMM.
//
// "Scalable Pretraining of Large MoE LMs on Aurora Super Computer", §3.1
// (stage 4) concatenates the weights of one projection over all experts of
// a rank into one tensor so that one grouped GEMM covers every expert.  The
// tensor-core GEMM here reads both operands K-major, so each projection is
// stored transposed (one row of K weights per output column):
//   gate/up  [E, 2f, d]: for N tile n of width 2h (h = gate_up_half_tile(f)),
//            rows n*2h .. n*2h+h-1 are gate columns n*h .. n*h+h-1 and rows
//            n*2h+h .. n*2h+2h-1 the same up columns, so one accumulator tile
//            holds matching gate and up columns for the SwiGLU epilogue;
//   down     [E, d, f].
#include "common.cuh"
#include "internal.h"

namespace moe {

int gate_up_half_tile(int f) { return (f % 128 == 0) ? 128 : 64; }

namespace {

constexpr int kTile = 32;

// dst[map(c)][r] = src[r][c] for one matrix of `rows` x `cols`; dst rows have
// `rows` elements.  map(c) = (c / half) * 2 * half + shift + c % half, or c
// when half == 0.
__global__ void __launch_bounds__(kTile * 8)
transpose_kernel(const __nv_bfloat16* __restrict__ src, __nv_bfloat16* __restrict__ dst, int rows, int cols,
                 int64_t src_stride, int64_t dst_stride, int half, int shift) {
  __shared__ __nv_bfloat16 tile[kTile][kTile + 2];
  const int64_t m = blockIdx.z;
  const __nv_bfloat16* s = src + m * src_stride;
  __nv_bfloat16* o = dst + m * dst_stride;
  const int c0 = blockIdx.x * kTile, r0 = blockIdx.y * kTile;
  for (int i = threadIdx.y; i < kTile; i += 8) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[i][threadIdx.x] = s[static_cast<int64_t>(r) * cols + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < kTile; i += 8) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) {
      const int64_t dr = half ? (static_cast<int64_t>(c / half) * 2 * half + shift + c % half) : c;
      o[dr * rows + r] = tile[threadIdx.x][i];
    }
  }
}

}  // namespace

cudaError_t launch_pack_weights(const void* w_gate, const void* w_up, const void* w_down, int E, int d, int f,
                                void* packed, cudaStream_t stream) {
  const int h = gate_up_half_tile(f);
  auto* gu = static_cast<__nv_bfloat16*>(packed);
  auto* dn = gu + static_cast<int64_t>(E) * 2 * f * d;
  const dim3 block(kTile, 8);
  // gate/up: source [E][d][f] (rows d, cols f) -> [E][2f][d]
  const dim3 grid_gu((f + kTile - 1) / kTile, (d + kTile - 1) / kTile, E);
  transpose_kernel<<<grid_gu, block, 0, stream>>>(static_cast<const __nv_bfloat16*>(w_gate), gu, d, f,
                                                  static_cast<int64_t>(d) * f, static_cast<int64_t>(2) * f * d, h, 0);
  transpose_kernel<<<grid_gu, block, 0, stream>>>(static_cast<const __nv_bfloat16*>(w_up), gu, d, f,
                                                  static_cast<int64_t>(d) * f, static_cast<int64_t>(2) * f * d, h, h);
  // down: source [E][f][d] (rows f, cols d) -> [E][d][f]
  const dim3 grid_dn((d + kTile - 1) / kTile, (f + kTile - 1) / kTile, E);
  transpose_kernel<<<grid_dn, block, 0, stream>>>(static_cast<const __nv_bfloat16*>(w_down), dn, f, d,
                                                  static_cast<int64_t>(f) * d, static_cast<int64_t>(d) * f, 0, 0);
  return cudaGetLastError();
}

}  // namespace moe
