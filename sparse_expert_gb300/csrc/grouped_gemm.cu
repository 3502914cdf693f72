// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// "Scalable Pretraining of Large MoE LMs on Aurora Super Computer", §3.1,
// Algorithm 1, stage 4: the expert MLP of every expert is one grouped GEMM
// per projection over expert-contiguous rows, with boundaries given by the
// cumulative token counts:
//   gate_out = Grouped_mm(mlp_in, gate_weight); up_out likewise;
//   mul_out = Silu(gate_out) * up_out;  mlp_out = Grouped_mm(mul_out, down_weight).
// Here gate and up are one GEMM whose N tile holds matching gate and up
// columns, so SiLU(gate)*up is the epilogue of that GEMM (H is written once,
// in bf16); the down GEMM's epilogue multiplies each row by its gate.
//
// Scheduling follows "Training a 1T-Params MoE on EU public infrastructure",
// Dynamic tile scheduling in SonicMoE: persistent blocks take tiles from a
// shared atomic counter instead of a fixed per-block list, so blocks that
// start late (their SM busy with other work) do not hold up the GEMM.
//
// Block of 320 threads, one per SM:
//   warp 0   TMA producer: takes tile ids, streams A and B K-blocks into a
//            ring of shared-memory stages (128-byte swizzle);
//   warp 1   MMA issuer: one thread issues tcgen05.mma (M=128, N=BN, K=16)
//            into one of two TMEM accumulators (double buffered);
//   warps 2-9 epilogue: tcgen05.ld of the accumulator, fp32 math, bf16
//            stores; TMEM lane quadrant = warp % 4, and the two warps of a
//            quadrant take one half of the tile's columns each.
// Gathered A ("Training a 1T-Params MoE on EU public infrastructure", the
// SonicMoE kernel that runs the expert GEMMs on the token-dispatch layout
// without a permuted copy): the gate/up GEMM can take its A rows straight
// from the token matrix, row r of the grouped problem being token
// gather_rows[r] (src_token): four warps copy each tile row's 128 bytes per
// K block with 16-byte cp.async into the swizzled stage, signal the stage
// barrier on completion, and the MMA thread fences the generic-proxy writes
// before the tensor cores read them (the epilogue then has four warps).
// Tiles: BM=128 rows of one expert's group (the last tile of a group is
// partial; rows past the group are computed and not stored), BN columns of
// that expert's weights.  Tile t of the flat order walks experts in order,
// and inside an expert the N tiles in order, each over all M tiles of the
// group, so consecutive tiles share a weight tile in L2.
#include <cuda.h>

#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // 64 bf16 = 128 bytes: one swizzle row
constexpr int kPackHalf = 64;  // gate (then up) columns of one packed gate/up weight tile
constexpr int UMMA_K = 16;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kRing = 4;  // tile ids fetched ahead
constexpr int kStoreStageBytes = kEpiWarps * 32 * 64;  // epilogue store transpose, 2 KB per epilogue warp
// dynamic shared memory for stage buffers: 227 KB per block minus room for
// the alignment slack, barriers, two [E+1] tables (E <= 1024) and the
// epilogue store buffers
constexpr int kStageBudget = 227 * 1024 - 1024 - 1024 - 2 * 1025 * 4 - 16 - kStoreStageBytes;

template <int BN>
struct Cfg {
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = kStageBudget / kStageBytes > 8 ? 8 : kStageBudget / kStageBytes;
  static constexpr int kTmemCols = 2 * BN;  // two accumulators
  static constexpr uint32_t kIdesc = umma_idesc_bf16_f32(BM, BN);
};

struct Params {
  const int32_t* offsets;
  const int32_t* gather_rows;  // gathered A: source row of every row, or null
  int64_t P;                   // rows of the grouped problem
  int64_t a_rows;              // rows of the gathered source matrix
  const void* gather_src;      // the gathered source matrix [a_rows, K]
  const float* row_scale;
  __nv_bfloat16* out;
  int32_t* tile_counter;
  int32_t* status;
  int E;
  int K;
  int n_per_expert;
  int n_tiles;
  int b_block_rows;  // rows of one packed weight tile (BN, or 128 for gate/up)
  int out_cols;
};

struct Smem {
  uint64_t full[8], empty[8];
  uint64_t tfull[2], tempty[2];
  uint64_t rfull[kRing], rempty[kRing];
  uint64_t drain;
  int32_t ring[kRing];
  uint32_t tmem_base;
  int abort;
};

// Gathered A: one 16-byte piece of a row, 16 bytes from src or zeros when
// src_bytes is 0 (a row past the problem).
__device__ __forceinline__ void cp_async_16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}

// One arrival on `bar` once every cp.async issued so far by this thread has
// landed (the arrival is expected in the barrier's count).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

template <int BN, bool kSwiGLU, bool kGather>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const Params p) {
  using C = Cfg<BN>;
  // gathered A: warps 2-5 are the epilogue and warps 6-9 fetch the A rows
  // (one thread per tile row); otherwise warps 2-9 are the epilogue
  constexpr int kEpi = kGather ? 4 : kEpiWarps;
  constexpr int kGatherThreads = kGather ? 128 : 0;
  const __nv_bfloat16* x_src = reinterpret_cast<const __nv_bfloat16*>(p.gather_src);
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  // stage buffers need 1024-byte alignment for the 128-byte swizzle
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + C::kStages * C::kABytes;
  Smem* S = reinterpret_cast<Smem*>(sB + C::kStages * C::kBBytes);
  int32_t* s_off = reinterpret_cast<int32_t*>(S + 1);  // [E+1] group boundaries
  int32_t* s_pre = s_off + (p.E + 1);                 // [E+1] M-tile prefix
  // [epilogue warps][32 rows][4 x 16 bytes] store transpose buffers
  uint4* s_stage = reinterpret_cast<uint4*>((reinterpret_cast<uintptr_t>(s_pre + p.E + 1) + 15) & ~uintptr_t(15));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &S->abort;

  // ---- set-up: group boundaries and M-tile prefix in shared memory
  if (warp == 0) {
    int carry = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      int lo = 0, hi = 0;
      if (e < p.E) {
        lo = __ldg(p.offsets + e);
        hi = __ldg(p.offsets + e + 1);
        s_off[e] = lo;
        if (e == p.E - 1) s_off[p.E] = hi;
      }
      int v = (hi - lo + BM - 1) / BM;
#pragma unroll
      for (int s = 1; s < 32; s <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, s);
        if (lane >= s) v += o;
      }
      if (e < p.E) s_pre[e + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) s_pre[0] = 0;
  } else if (warp == 1) {
    tmem_alloc(&S->tmem_base, C::kTmemCols);
    tmem_relinquish();
  } else if (warp == 2 && lane == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&S->full[i], 1 + kGatherThreads);
      mbar_init(&S->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S->tfull[i], 1);
      mbar_init(&S->tempty[i], kEpi);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&S->rfull[i], 1);
      mbar_init(&S->rempty[i], 1 + kEpi + kGatherThreads / 32);
    }
    mbar_init(&S->drain, 1);
    S->abort = 0;
    fence_barrier_init();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const int total_tiles = s_pre[p.E] * p.n_tiles;
  const int num_kb = (p.K + BK - 1) / BK;
  const uint32_t tmem_base = S->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_a);
      tma_prefetch_desc(&tm_b);
      int stage = 0;
      uint32_t phase = 0;
      int rs = 0;
      uint32_t rphase = 0;
      bool ok = true;
      int last_stage = -1;
      uint32_t last_phase = 0;
      for (;;) {
        if (!mbar_wait(&S->rempty[rs], rphase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        int t = atomicAdd(p.tile_counter, 1);
        if (t >= total_tiles) t = -1;
        S->ring[rs] = t;
        mbar_arrive(&S->rfull[rs]);
        if (++rs == kRing) {
          rs = 0;
          rphase ^= 1u;
        }
        if (t < 0) break;
        int e, mt, nt;
        decode_tile(t, s_pre, p.E, p.n_tiles, e, mt, nt);
        const int row0 = s_off[e] + mt * BM;
        // weight tiles are stored tile-major: block (e, tile, kb) is
        // b_block_rows x 64, and an N tile spans BN / b_block_rows of them
        const int per_tile = BN / p.b_block_rows;
        const int bblk = (e * p.n_tiles + nt) * per_tile * num_kb;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&S->empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          if constexpr (kGather) {
            mbar_arrive_expect_tx(&S->full[stage], C::kBBytes);
          } else {
            mbar_arrive_expect_tx(&S->full[stage], C::kStageBytes);
            tma_load_2d(sA + stage * C::kABytes, &tm_a, &S->full[stage], kb * BK, row0);
          }
          for (int j = 0; j < per_tile; ++j)
            tma_load_3d(sB + stage * C::kBBytes + j * p.b_block_rows * BK * 2, &tm_b, &S->full[stage], 0, 0,
                        bblk + j * num_kb + kb);
          last_stage = stage;
          last_phase = phase;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (!ok) {
        record_status(p.status, kStatusTimeout);
        *abort_flag = 1;
        // let the last copy land before the block can exit
        if (last_stage >= 0) {
          volatile int never = 0;
          mbar_wait(&S->full[last_stage], last_phase, &never);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int rs = 0;
      uint32_t rphase = 0;
      int acc = 0;
      uint32_t aphase = 0;
      bool ok = true;
      for (;;) {
        if (!mbar_wait(&S->rfull[rs], rphase, abort_flag)) {
          ok = false;
          break;
        }
        const int t = S->ring[rs];
        mbar_arrive(&S->rempty[rs]);
        if (++rs == kRing) {
          rs = 0;
          rphase ^= 1u;
        }
        if (t < 0) break;
        if (!mbar_wait(&S->tempty[acc], aphase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&S->full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          // gathered A rows were written by the gather threads' copies
          // (generic proxy); order them before the tensor cores read them
          if constexpr (kGather) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          tc_fence_after_sync();
          // the stage's descriptors once; a K step of 16 advances the start
          // address (16-byte units) by 2
          const uint64_t da = sw128_kmajor_desc(smem_addr(sA + stage * C::kABytes));
          const uint64_t db = sw128_kmajor_desc(smem_addr(sB + stage * C::kBBytes));
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk)
            umma_bf16(d_tmem, da + 2 * kk, db + 2 * kk, C::kIdesc, (kb | kk) != 0 ? 1u : 0u);
          umma_commit(&S->empty[stage]);  // frees the stage when these MMAs finish
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&S->tfull[acc]);  // accumulator ready for the epilogue
        acc ^= 1;
        if (acc == 0) aphase ^= 1u;
      }
      if (!ok) {
        record_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // every MMA issued by this thread has completed once drain flips
      umma_commit(&S->drain);
      volatile int never = 0;
      mbar_wait(&S->drain, 0, &never);
    }
  } else if (kGather && warp >= 2 + kEpi) {
    // ------------------------------------------- gathered A rows (4 warps)
    // thread g fetches row g of every A tile: token gather_rows[row], its 64
    // columns of this K block as 8 copies of 16 bytes into the swizzled row
    // (piece j at slot j ^ (g % 8)); rows past the problem read as zeros
    const int g = threadIdx.x - 32 * (2 + kEpi);
    int stage = 0;
    uint32_t phase = 0;
    int rs = 0;
    uint32_t rphase = 0;
    bool ok = true;
    for (;;) {
      if (!mbar_wait_warp(&S->rfull[rs], rphase, abort_flag)) {
        ok = false;
        break;
      }
      const int t = S->ring[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(&S->rempty[rs]);
      if (++rs == kRing) {
        rs = 0;
        rphase ^= 1u;
      }
      if (t < 0) break;
      int e, mt, nt;
      decode_tile(t, s_pre, p.E, p.n_tiles, e, mt, nt);
      const int64_t row = static_cast<int64_t>(s_off[e]) + mt * BM + g;
      // a source token outside [0, a_rows) (a row the dispatch pass left
      // unwritten) is read as zeros, never as an address
      const int64_t tok = row < p.P ? static_cast<int64_t>(__ldg(p.gather_rows + row)) : -1;
      const bool tok_ok = tok >= 0 && tok < p.a_rows;
      const int src_bytes = tok_ok ? 16 : 0;
      const __nv_bfloat16* src_row = x_src + (tok_ok ? tok * p.K : 0);
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait_warp(&S->empty[stage], phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* dst = sA + stage * C::kABytes + g * 128;
        const __nv_bfloat16* src = src_row + kb * BK;
#pragma unroll
        for (int j = 0; j < 8; ++j) cp_async_16(dst + ((j ^ (g & 7)) << 4), src + j * 8, src_bytes);
        cp_async_arrive(&S->full[stage]);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
    // no copy of this thread may still be in flight when the block exits
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (!ok && lane == 0) {
      record_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int quad = warp & 3;         // TMEM lanes 32*quad .. 32*quad+31
    const int half = (warp - 2) >> 2;  // which half of the tile's columns (0 with 4 epilogue warps)
    uint4* sbuf = s_stage + (warp - 2) * 32 * 4;
    int rs = 0;
    uint32_t rphase = 0;
    int acc = 0;
    uint32_t aphase = 0;
    for (;;) {
      if (!mbar_wait_warp(&S->rfull[rs], rphase, abort_flag)) break;
      const int t = S->ring[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(&S->rempty[rs]);
      if (++rs == kRing) {
        rs = 0;
        rphase ^= 1u;
      }
      if (t < 0) break;
      int e, mt, nt;
      decode_tile(t, s_pre, p.E, p.n_tiles, e, mt, nt);
      // this warp's 32 rows of the tile start at global row wrow0
      const int64_t wrow0 = static_cast<int64_t>(s_off[e]) + mt * BM + quad * 32;
      const int valid_rows = static_cast<int>(min(static_cast<int64_t>(32), max(static_cast<int64_t>(0),
                                                                                 s_off[e + 1] - wrow0)));
      if (!mbar_wait_warp_suspend(&S->tfull[acc], aphase, abort_flag)) {
        if (lane == 0) {
          record_status(p.status, kStatusTimeout);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after_sync();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
      // hands the accumulator back to the MMA warp once this warp has read
      // its last columns (the stores of the last chunk still follow)
      auto release_accumulator = [&]() {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S->tempty[acc]);
      };
      if constexpr (kSwiGLU) {
        // the tile's output features [nt * H, nt * H + H) come from packed
        // gate/up tiles of 64 gate then the same 64 up columns
        constexpr int H = BN / 2;
        constexpr int kCols = H / (kEpi / 4);
        const int c0 = half * kCols;
        __nv_bfloat16* dst = p.out + wrow0 * p.out_cols + static_cast<int64_t>(nt) * H + c0;
#pragma unroll 1
        for (int c = 0; c < kCols; c += 32) {
          uint32_t g[32], u[32];
          const int o = c0 + c;
          const int gcol = (o / kPackHalf) * 2 * kPackHalf + o % kPackHalf;
          tmem_ld_32x32(taddr + gcol, g);
          tmem_ld_32x32(taddr + gcol + kPackHalf, u);
          tmem_ld_wait();
          if (c + 32 == kCols) release_accumulator();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float h0 = silu_f32(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
            const float h1 = silu_f32(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
            packed[i] = pack_bf16x2(h0, h1);
          }
          store_chunk_coalesced(packed, sbuf, lane, dst + c, p.out_cols, valid_rows);
        }
      } else {
        constexpr int kCols = BN / (kEpi / 4);
        const int c0 = half * kCols;
        const float scale = (lane < valid_rows && p.row_scale != nullptr) ? __ldg(p.row_scale + wrow0 + lane) : 1.0f;
        __nv_bfloat16* dst = p.out + wrow0 * p.out_cols + static_cast<int64_t>(nt) * BN + c0;
#pragma unroll 1
        for (int c = 0; c < kCols; c += 32) {
          uint32_t v[32];
          tmem_ld_32x32(taddr + c0 + c, v);
          tmem_ld_wait();
          if (c + 32 == kCols) release_accumulator();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[i] = pack_bf16x2(scale * __uint_as_float(v[2 * i]), scale * __uint_as_float(v[2 * i + 1]));
          store_chunk_coalesced(packed, sbuf, lane, dst + c, p.out_cols, valid_rows);
        }
      }
      acc ^= 1;
      if (acc == 0) aphase ^= 1u;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------ host side
template <int BN, bool kSwiGLU, bool kGather>
cudaError_t launch_bn(const GroupedGemmProblem& pb, int num_sms, cudaStream_t stream) {
  using C = Cfg<BN>;
  CUtensorMap ma, mb;
  // the gathered variant reads A with plain copies; its map is unused (built over the same matrix)
  if (!make_bf16_map_2d(&ma, pb.a, kGather ? pb.a_rows : pb.P, pb.K, BK, kGather ? 1 : BM))
    return cudaErrorInvalidValue;
  // tile-major weights as [blocks][block rows][64], one block per box
  const int block_rows = kSwiGLU ? 2 * kPackHalf : BN;
  const int64_t blocks = static_cast<int64_t>(pb.E) * (pb.n_per_expert / block_rows) * ((pb.K + BK - 1) / BK);
  if (!make_bf16_map_3d(&mb, pb.b, BK, block_rows, blocks, BK, block_rows)) return cudaErrorInvalidValue;
  Params prm;
  prm.offsets = pb.offsets;
  prm.gather_rows = pb.gather_rows;
  prm.P = pb.P;
  prm.a_rows = pb.a_rows;
  prm.gather_src = pb.a;
  prm.row_scale = pb.row_scale;
  prm.out = static_cast<__nv_bfloat16*>(pb.out);
  prm.tile_counter = pb.tile_counter;
  prm.status = pb.status;
  prm.E = pb.E;
  prm.K = pb.K;
  prm.n_per_expert = pb.n_per_expert;
  prm.n_tiles = pb.n_per_expert / BN;
  prm.b_block_rows = block_rows;
  prm.out_cols = pb.out_cols;
  const size_t smem = 1024 + static_cast<size_t>(C::kStages) * C::kStageBytes + sizeof(Smem) +
                      2 * static_cast<size_t>(pb.E + 1) * sizeof(int32_t) + 16 + kStoreStageBytes;
  auto kernel = grouped_gemm_kernel<BN, kSwiGLU, kGather>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  // persistent: one block per SM, never more blocks than an upper bound on tiles
  const int64_t max_tiles = (pb.P / BM + pb.E) * static_cast<int64_t>(prm.n_tiles);
  const int grid = static_cast<int>(max_tiles < num_sms ? max_tiles : num_sms);
  kernel<<<grid, kThreads, smem, stream>>>(ma, mb, prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm(const GroupedGemmProblem& pb, Epilogue epi, int num_sms, cudaStream_t stream) {
  if (pb.P == 0) return cudaSuccess;
  // SM pairs with the weights as the 256-row operand where the weight rows
  // per expert are a multiple of 256 (grouped_gemm_2sm.cu)
  if (pb.gather_rows == nullptr && grouped_gemm_2sm_supported(pb, epi))
    return launch_grouped_gemm_2sm(pb, epi, num_sms, stream);
  if (epi == Epilogue::kSwiGLU) {
    // N tile = one or two packed gate/up tiles (64 gate + 64 up columns each)
    if (gate_up_half_tile(pb.out_cols) != kPackHalf) return cudaErrorNotSupported;
    const bool wide = pb.n_per_expert % 256 == 0;
    if (pb.gather_rows != nullptr)
      return wide ? launch_bn<256, true, true>(pb, num_sms, stream) : launch_bn<128, true, true>(pb, num_sms, stream);
    return wide ? launch_bn<256, true, false>(pb, num_sms, stream) : launch_bn<128, true, false>(pb, num_sms, stream);
  }
  if (pb.gather_rows != nullptr) return cudaErrorNotSupported;
  // N tile of the packed down weights
  switch (down_tile_n(pb.out_cols)) {
    case 256: return launch_bn<256, false, false>(pb, num_sms, stream);
    case 128: return launch_bn<128, false, false>(pb, num_sms, stream);
    default: return launch_bn<64, false, false>(pb, num_sms, stream);
  }
}

}  // namespace moe
