// Device helpers shared by the grouped GEMM kernels.
#pragma once

#include "common.cuh"

namespace moe {

// Expert, M tile and N tile of flat tile t.  s_pre[e] = M tiles of experts
// before e (s_pre[E] = all).  The largest e with s_pre[e]*nt <= t has a
// non-empty range containing t.
__device__ __forceinline__ void decode_tile(int t, const int32_t* s_pre, int E, int n_tiles, int& e, int& mt,
                                            int& nt) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pre[mid] * n_tiles <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  e = lo;
  const int mtiles = s_pre[e + 1] - s_pre[e];
  const int local = t - s_pre[e] * n_tiles;
  nt = local / mtiles;
  mt = local - nt * mtiles;
}

// Stores one 32-column chunk of the epilogue warp's 32 tile rows.  Thread
// `lane` holds row `lane` as 16 packed bf16x2 words (64 bytes).  Through a
// 2 KB shared-memory transpose, each 16-byte global store instruction then
// covers 8 rows x 64 contiguous bytes instead of 32 rows x 16 bytes.  In
// the buffer, 16-byte piece j of row r sits at slot j ^ ((r >> 1) & 3),
// so the row-wise writes and the row-pair reads are free of bank
// conflicts.  Rows at or past `valid_rows` are not stored.
__device__ __forceinline__ void store_chunk_coalesced(const uint32_t (&w)[16], uint4* sbuf, int lane,
                                                      __nv_bfloat16* row0, int64_t ld, int valid_rows) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    sbuf[lane * 4 + (j ^ ((lane >> 1) & 3))] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = i * 8 + (lane >> 2);
    const int g = lane & 3;
    const uint4 v = sbuf[r * 4 + (g ^ ((r >> 1) & 3))];
    if (r < valid_rows) *reinterpret_cast<uint4*>(row0 + r * ld + g * 8) = v;
  }
  __syncwarp();
}

// Inverse of store_chunk_coalesced: loads 32 rows x 32 bf16 (64 bytes a
// row) starting at row0 with row stride ld, 8 rows x 64 contiguous bytes per
// 16-byte load instruction, and hands row `lane` to thread `lane` as 16
// packed bf16x2 words.  Rows at or past `valid_rows` read as zero.
__device__ __forceinline__ void load_chunk_coalesced(uint32_t (&w)[16], uint4* sbuf, int lane,
                                                     const __nv_bfloat16* row0, int64_t ld, int valid_rows) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = i * 8 + (lane >> 2);
    const int g = lane & 3;
    const uint4 v = r < valid_rows ? *reinterpret_cast<const uint4*>(row0 + r * ld + g * 8) : make_uint4(0, 0, 0, 0);
    sbuf[r * 4 + (g ^ ((r >> 1) & 3))] = v;
  }
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 v = sbuf[lane * 4 + (j ^ ((lane >> 1) & 3))];
    w[4 * j] = v.x;
    w[4 * j + 1] = v.y;
    w[4 * j + 2] = v.z;
    w[4 * j + 3] = v.w;
  }
  __syncwarp();
}

}  // namespace moe
