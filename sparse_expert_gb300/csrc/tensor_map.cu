// Tiled bf16 tensor maps for the TMA loads of the GEMM kernels.  The driver
// entry point is fetched through the runtime, so the library needs no link
// against libcuda.
#include <cuda.h>

#include "internal.h"

namespace moe {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

bool encode(CUtensorMap* map, const void* ptr, cuuint32_t rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
            CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, type, rank, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool make_bf16_map_2d(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_cols, int box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  return encode(map, ptr, 2, dims, strides, box);
}

// The same with 64-byte swizzling (boxes of 32 bf16 columns): the 16-byte
// pieces of row r of a 512-byte atom are permuted by (r >> 1) & 3.
bool make_bf16_map_2d_sw64(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_cols,
                           int box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  return encode(map, ptr, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

bool make_bf16_map_3d(CUtensorMap* map, const void* ptr, int64_t d0, int64_t d1, int64_t d2, int box0, int box1,
                      int box2) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d0), static_cast<cuuint64_t>(d1), static_cast<cuuint64_t>(d2)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d0) * 2, static_cast<cuuint64_t>(d0 * d1) * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box0), static_cast<cuuint32_t>(box1),
                             static_cast<cuuint32_t>(box2)};
  return encode(map, ptr, 3, dims, strides, box);
}

// A row-major [rows, cols] matrix seen as (64 columns, rows, cols / 64
// column blocks): the block stride (128 bytes) is below the row stride, so
// one box of (64, box_rows, box_blocks) lands in shared memory as
// box_blocks consecutive [box_rows][64] chunks, each in the 128-byte
// swizzled MN-major layout the MMA descriptors read.
bool make_bf16_map_col_blocks(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_rows,
                              int box_blocks) {
  if (cols % 64 != 0) return false;
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, 128};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(box_blocks)};
  return encode(map, ptr, 3, dims, strides, box);
}

// A stack of packed gate/up blocks of [128 rows][64 columns] (rows 0-63
// gate features, 64-127 the same up features) seen as (64 columns, 16 rows,
// 2 halves, 8 * blocks groups of 16 rows): the half stride (64 rows) lies
// above the group stride (16 rows), so one box of (64, 16, 2, 4) at group
// 8 * block lands a block in shared memory with its rows reordered as
// [group][half][row]: each 32-row quarter holds 16 gate features followed
// by the same 16 up features.
bool make_bf16_map_gate_up_quads(CUtensorMap* map, const void* ptr, int64_t blocks) {
  const cuuint64_t dims[4] = {64, 16, 2, static_cast<cuuint64_t>(blocks) * 8};
  const cuuint64_t strides[3] = {128, 64 * 128, 16 * 128};
  const cuuint32_t box[4] = {64, 16, 2, 4};
  return encode(map, ptr, 4, dims, strides, box);
}

bool make_u8_map_rows64_sw64(CUtensorMap* map, const void* ptr, int64_t rows, int box_rows) {
  const cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {64};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  return encode(map, ptr, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

}  // namespace moe
