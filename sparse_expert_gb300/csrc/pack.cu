// One-time layout transform of the expert weights for the grouped GEMM.
//
// "Scalable Pretraining of Large MoE LMs on Aurora Super Computer", §3.1
// (stage 4) concatenates the weights of one projection over all experts of
// a rank into one tensor so that one grouped GEMM covers every expert.  The
// tensor-core GEMM here reads both operands K-major, so each projection is
// stored transposed (K weights per output column), and tile-major, so that
// the B operand of one GEMM stage (BN output columns x 64 K values) is one
// contiguous block of BN * 128 bytes and every weight load streams whole
// DRAM pages:
//   element (e, n, k) of a projection with N tile BN and K = 64 * num_kb
//   sits at (((e * n_tiles + n / BN) * num_kb + k / 64) * BN + n % BN) * 64
//   + k % 64.
//   gate/up  N = 2f, K = d, BN = 2h (h = gate_up_half_tile(f)): in N tile t,
//            rows 0 .. h-1 are gate columns t*h .. t*h+h-1 and rows
//            h .. 2h-1 the same up columns, so one accumulator tile holds
//            matching gate and up columns for the SwiGLU epilogue;
//   down     N = d, K = f, BN = down_tile_n(d).
#include "common.cuh"
#include "internal.h"

namespace moe {

// 64 gate then 64 up columns per packed tile: a 256-row tile of the paired
// GEMM is two packed tiles, one per SM, each holding matching gate and up rows
int gate_up_half_tile(int f) { (void)f; return 64; }
int gate_up_tile_n(int f) { return 2 * gate_up_half_tile(f); }
int down_tile_n(int d) { return d % 256 == 0 ? 256 : d % 128 == 0 ? 128 : 64; }

namespace {

constexpr int kTile = 32;

// One matrix src[r][c] (rows = K, cols) goes to packed element (n, k) =
// (map(c), r) of the tile-major layout above, with map(c) =
// (c / half) * 2 * half + shift + c % half, or c when half == 0.
__global__ void __launch_bounds__(kTile * 8)
transpose_kernel(const __nv_bfloat16* __restrict__ src, __nv_bfloat16* __restrict__ dst, int rows, int cols,
                 int64_t src_stride, int64_t dst_stride, int half, int shift, int bn) {
  __shared__ __nv_bfloat16 tile[kTile][kTile + 2];
  const int64_t m = blockIdx.z;
  const __nv_bfloat16* s = src + m * src_stride;
  __nv_bfloat16* o = dst + m * dst_stride;
  const int num_kb = rows / 64;
  const int c0 = blockIdx.x * kTile, r0 = blockIdx.y * kTile;
  for (int i = threadIdx.y; i < kTile; i += 8) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[i][threadIdx.x] = s[static_cast<int64_t>(r) * cols + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < kTile; i += 8) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) {
      const int64_t n = half ? (static_cast<int64_t>(c / half) * 2 * half + shift + c % half) : c;
      const int64_t off = (((n / bn) * num_kb + r / 64) * bn + n % bn) * 64 + r % 64;
      o[off] = tile[threadIdx.x][i];
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
  // gate/up: source [E][d][f] (rows d = K, cols f)
  const dim3 grid_gu((f + kTile - 1) / kTile, (d + kTile - 1) / kTile, E);
  transpose_kernel<<<grid_gu, block, 0, stream>>>(static_cast<const __nv_bfloat16*>(w_gate), gu, d, f,
                                                  static_cast<int64_t>(d) * f, static_cast<int64_t>(2) * f * d, h, 0,
                                                  2 * h);
  transpose_kernel<<<grid_gu, block, 0, stream>>>(static_cast<const __nv_bfloat16*>(w_up), gu, d, f,
                                                  static_cast<int64_t>(d) * f, static_cast<int64_t>(2) * f * d, h, h,
                                                  2 * h);
  // down: source [E][f][d] (rows f = K, cols d)
  const dim3 grid_dn((d + kTile - 1) / kTile, (f + kTile - 1) / kTile, E);
  transpose_kernel<<<grid_dn, block, 0, stream>>>(static_cast<const __nv_bfloat16*>(w_down), dn, f, d,
                                                  static_cast<int64_t>(f) * d, static_cast<int64_t>(d) * f, 0, 0,
                                                  down_tile_n(d));
  return cudaGetLastError();
}

}  // namespace moe
