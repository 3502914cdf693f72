// Grouped expert GEMMs of the backward pass on the tensor cores (tcgen05,
// sm_103a).
//
// "Scalable Pretraining of Large MoE LMs on Aurora Super Computer", §3.1,
// Algorithm 1, stage 4 (gate/up grouped GEMMs, Silu(gate)*up, down grouped
// GEMM), differentiated.  With G, U the gate and up pre-activations of a row,
// H = Silu(G)*U and dY the gradient of the row's expert output:
//   dH = dY Wd^T,   dG = dH U Silu'(G),   dU = dH Silu(G),
//   dX = dG Wg^T + dU Wu^T,
//   dWd[e] = H_e^T dY_e,   dWg[e] = X_e^T dG_e,   dWu[e] = X_e^T dU_e.
// One kernel template covers four GEMMs (Mode):
//   kGateUpSave   the forward gate/up GEMM that also stores G and U (bf16),
//                 the activations the backward reads;
//   kDgradSwiGLU  dY x Wd -> dH, with dG and dU formed in the epilogue;
//   kDgradPlain   [dG | dU] x [Wg ; Wu] -> dX;
//   kWgrad        a weight gradient: for each expert, the contraction runs
//                 over that expert's rows (K-grouped).
// The first three are M-grouped like the forward (128-row tiles inside one
// expert's group).  The dgrad GEMMs read the forward's tile-major packed
// weights transposed: the contraction runs along the packed rows, so B is
// MN-major in shared memory, staged as 64 x 64 chunks of one packed block.
// The weight-gradient GEMM reads both operands row by row (MN-major chunks)
// and zeroes, in shared memory, the rows of an expert's last K block that
// belong to the next expert before the tensor cores read them.
// G, U, dG and dU are stored interleaved like the packed gate/up weights:
// N tile t of the gate/up GEMM holds gate columns t*h .. t*h+h-1, then the
// same up columns (2h per tile).
//
// Block of 320 threads, one per SM, the same roles as the forward kernel:
// warp 0 TMA producer, warp 1 MMA issuer (the whole warp waits; lane 0
// issues; in kWgrad the warp zeroes the rows past the expert), warps 2-9
// epilogue.  Tiles come from a shared atomic counter (dynamic scheduling).
#include <cuda.h>

#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // 64 bf16 = 128 bytes: one swizzle row
constexpr int UMMA_K = 16;
constexpr int kChunk = 64 * 64 * 2;  // one 64 x 64 bf16 chunk (MN-major staging)
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kRing = 4;
constexpr int kStoreStageBytes = kEpiWarps * 32 * 64;
constexpr int kStageBudget = 227 * 1024 - 1024 - 1024 - 2 * 1025 * 4 - 1024 - kStoreStageBytes;
// weight gradients: 64-column chunks whose rows past an expert's last row are
// zeroed before the last K block's MMAs (A's: BM / 64 of them)
constexpr int kZeroChunks = BM / 64;

enum class Mode { kGateUpSave, kDgradSwiGLU, kDgradPlain, kWgrad };

template <int BN, Mode M>
struct Cfg {
  static constexpr bool kAMN = (M == Mode::kWgrad);
  static constexpr bool kBMN = (M != Mode::kGateUpSave);
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = kStageBudget / kStageBytes > 8 ? 8 : kStageBudget / kStageBytes;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr uint32_t kIdesc = umma_idesc_bf16_f32_major(BM, BN, kAMN, kBMN);
};

struct Params {
  const int32_t* offsets;
  int32_t* tile_counter;
  int32_t* status;
  int E;
  int K;          // contraction length of the M-grouped modes
  int n_tiles;    // N tiles per expert
  int m_tiles;    // kWgrad: M tiles per expert
  int M_ext;      // kWgrad: rows of one expert's gradient
  int N_ext;      // N extent
  int b_rows;     // dgrad: rows of one packed weight block (the forward's N tile)
  int b_tiles;    // dgrad: packed N tiles per expert
  int b_kblocks;  // dgrad: packed K blocks per N tile
  int half;       // h: gate (and up) columns per interleaved gate/up tile
  int interleaved;               // kWgrad: N runs over interleaved gate/up columns
  const __nv_bfloat16* gu;       // kDgradSwiGLU: G, U [P, 2f]
  __nv_bfloat16* out;            // H | dG,dU | dX | dWd or dWg
  __nv_bfloat16* out2;           // kGateUpSave: G,U;  kWgrad interleaved: dWu
  int out_cols;                  // row stride of out (and of out2)
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

// Tile t of a weight-gradient GEMM: expert, M tile, N tile (M fastest).
__device__ __forceinline__ void decode_wgrad(int t, int m_tiles, int n_tiles, int& e, int& mt, int& nt) {
  const int per = m_tiles * n_tiles;
  e = t / per;
  const int local = t - e * per;
  nt = local / m_tiles;
  mt = local - nt * m_tiles;
}

template <int BN, Mode M>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_bwd_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                        const __grid_constant__ CUtensorMap tm_o1, const __grid_constant__ CUtensorMap tm_o2,
                        const Params p) {
  using C = Cfg<BN, M>;
  constexpr bool kW = (M == Mode::kWgrad);
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + C::kStages * C::kABytes;
  Smem* S = reinterpret_cast<Smem*>(sB + C::kStages * C::kBBytes);
  int32_t* s_off = reinterpret_cast<int32_t*>(S + 1);  // [E+1] group boundaries
  int32_t* s_pre = s_off + (p.E + 1);                 // [E+1] M-tile prefix (M-grouped modes)
  // per epilogue warp 2 KB of store staging, 1024-byte aligned (the 64-byte
  // swizzle of the weight gradients' TMA stores repeats every 512 bytes)
  uint4* s_stage =
      reinterpret_cast<uint4*>((reinterpret_cast<uintptr_t>(s_pre + p.E + 1) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &S->abort;

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
      mbar_init(&S->full[i], 1);
      mbar_init(&S->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S->tfull[i], 1);
      mbar_init(&S->tempty[i], kEpiWarps);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&S->rfull[i], 1);
      mbar_init(&S->rempty[i], 1 + kEpiWarps);
    }
    mbar_init(&S->drain, 1);
    S->abort = 0;
    fence_barrier_init();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const int total_tiles = kW ? p.E * p.m_tiles * p.n_tiles : s_pre[p.E] * p.n_tiles;
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
        int e, mt, nt, row0, num_kb;
        if constexpr (kW) {
          decode_wgrad(t, p.m_tiles, p.n_tiles, e, mt, nt);
          row0 = s_off[e];
          num_kb = (s_off[e + 1] - row0 + BK - 1) / BK;
        } else {
          decode_tile(t, s_pre, p.E, p.n_tiles, e, mt, nt);
          row0 = s_off[e] + mt * BM;
          num_kb = p.K / BK;
        }
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&S->empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = sA + stage * C::kABytes;
          uint8_t* b_dst = sB + stage * C::kBBytes;
          mbar_arrive_expect_tx(&S->full[stage], C::kStageBytes);
          if constexpr (kW) {
            // rows row0 + kb*64 .. +63 of both operands: one copy per operand
            // of BM / 64 (BN / 64) consecutive 64-column chunks
            tma_load_3d(a_dst, &tm_a, &S->full[stage], 0, row0 + kb * BK, mt * (BM / 64));
            tma_load_3d(b_dst, &tm_b, &S->full[stage], 0, row0 + kb * BK, nt * (BN / 64));
          } else {
            tma_load_2d(a_dst, &tm_a, &S->full[stage], kb * BK, row0);
            if constexpr (M == Mode::kGateUpSave) {
              tma_load_3d(b_dst, &tm_b, &S->full[stage], 0, 0, (e * p.n_tiles + nt) * (p.K / BK) + kb);
            } else {
              // K rows kb*64.. of this expert's weights are rows of packed
              // N tile (kb*64)/b_rows; N chunk c is that tile's K block
              // nt*BN/64 + c: one copy of BN / 64 consecutive blocks
              const int kr = kb * BK;
              const int blk0 = (e * p.b_tiles + kr / p.b_rows) * p.b_kblocks + nt * (BN / 64);
              const int brow = kr % p.b_rows;
              tma_load_3d(b_dst, &tm_b, &S->full[stage], 0, brow, blk0);
            }
          }
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
        if (last_stage >= 0) {
          volatile int never = 0;
          mbar_wait(&S->full[last_stage], last_phase, &never);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int rs = 0;
    uint32_t rphase = 0;
    int acc = 0;
    uint32_t aphase = 0;
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
      int num_kb, rows = 0;
      if constexpr (kW) {
        int e, mt, nt;
        decode_wgrad(t, p.m_tiles, p.n_tiles, e, mt, nt);
        rows = s_off[e + 1] - s_off[e];
        num_kb = (rows + BK - 1) / BK;
      } else {
        num_kb = p.K / BK;
      }
      if (!mbar_wait_warp(&S->tempty[acc], aphase ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait_warp(&S->full[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint8_t* a_st = sA + stage * C::kABytes;
        uint8_t* b_st = sB + stage * C::kBBytes;
        // MMAs of 16 K rows each; in an expert's last K block only those
        // holding its rows run (kWgrad)
        int n_kk = BK / UMMA_K;
        if constexpr (kW) {
          const int valid = rows - kb * BK;
          if (valid < BK) {
            n_kk = (valid + UMMA_K - 1) / UMMA_K;
            const int zend = n_kk * UMMA_K;
            if (valid < zend) {
              // rows valid .. zend-1 belong to the next expert (or lie past
              // the matrix, where TMA filled zeros): zeroing them in A's
              // chunks alone removes their products, since B's rows there are
              // finite; a whole 128-byte row is zero whatever the swizzle
              // does inside it
              // lane: 16-byte piece lane % 8 of rows valid + lane / 8, +4, ...
              const uint4 zero = make_uint4(0, 0, 0, 0);
              const int piece = lane & 7;
#pragma unroll
              for (int c = 0; c < kZeroChunks; ++c) {
                uint8_t* cb = c < BM / 64 ? a_st + c * kChunk : b_st + (c - BM / 64) * kChunk;
                for (int r = valid + (lane >> 3); r < zend; r += 4) reinterpret_cast<uint4*>(cb + r * 128)[piece] = zero;
              }
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            __syncwarp();
          }
        }
        if (lane == 0) {
          // the stage's descriptors once; a K step of 16 advances the start
          // address (16-byte units) by 2 (K-major) or 16 rows of 128 bytes (MN-major)
          const uint64_t da0 = C::kAMN ? sw128_mnmajor_desc(smem_addr(a_st), kChunk) : sw128_kmajor_desc(smem_addr(a_st));
          const uint64_t db0 = C::kBMN ? sw128_mnmajor_desc(smem_addr(b_st), kChunk) : sw128_kmajor_desc(smem_addr(b_st));
          constexpr uint64_t kStepA = C::kAMN ? (UMMA_K * 128) >> 4 : (UMMA_K * 2) >> 4;
          constexpr uint64_t kStepB = C::kBMN ? (UMMA_K * 128) >> 4 : (UMMA_K * 2) >> 4;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            if (kk >= n_kk) break;
            umma_bf16(d_tmem, da0 + kk * kStepA, db0 + kk * kStepB, C::kIdesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(&S->empty[stage]);
        }
        __syncwarp();
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(&S->tfull[acc]);  // (at once when the tile had no rows)
      __syncwarp();
      acc ^= 1;
      if (acc == 0) aphase ^= 1u;
    }
    if (lane == 0) {
      if (!ok) {
        record_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      umma_commit(&S->drain);
      volatile int never = 0;
      mbar_wait(&S->drain, 0, &never);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int quad = warp & 3;
    const int halfc = (warp - 2) >> 2;
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
      int e, mt, nt, valid_rows, k_rows = 1;
      int64_t wrow0;
      if constexpr (kW) {
        decode_wgrad(t, p.m_tiles, p.n_tiles, e, mt, nt);
        k_rows = s_off[e + 1] - s_off[e];
        wrow0 = static_cast<int64_t>(mt) * BM + quad * 32;  // gradient row (M index)
        valid_rows = static_cast<int>(min(static_cast<int64_t>(32), max(static_cast<int64_t>(0), p.M_ext - wrow0)));
      } else {
        decode_tile(t, s_pre, p.E, p.n_tiles, e, mt, nt);
        wrow0 = static_cast<int64_t>(s_off[e]) + mt * BM + quad * 32;
        valid_rows = static_cast<int>(min(static_cast<int64_t>(32), max(static_cast<int64_t>(0),
                                                                        s_off[e + 1] - wrow0)));
      }
      if (!mbar_wait_warp_suspend(&S->tfull[acc], aphase, abort_flag)) {
        if (lane == 0) {
          record_status(p.status, kStatusTimeout);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after_sync();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
      auto release_accumulator = [&]() {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S->tempty[acc]);
      };
      if constexpr (M == Mode::kGateUpSave) {
        const int H = BN / 2;  // gate columns [0, H), up columns [H, 2H) of the accumulator
        const int kCols = H / 2;
        const int c0 = halfc * kCols;
        __nv_bfloat16* hdst = p.out + wrow0 * p.out_cols + static_cast<int64_t>(nt) * H + c0;
        __nv_bfloat16* gdst = p.out2 + wrow0 * (2 * p.out_cols) + static_cast<int64_t>(nt) * BN + c0;
#pragma unroll 1
        for (int c = 0; c < kCols; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld_32x32(taddr + c0 + c, g);
          tmem_ld_32x32(taddr + H + c0 + c, u);
          tmem_ld_wait();
          if (c + 32 == kCols) release_accumulator();
          uint32_t ph[16], pg[16], pu[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
            const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
            ph[i] = pack_bf16x2(silu_f32(g0) * u0, silu_f32(g1) * u1);
            pg[i] = pack_bf16x2(g0, g1);
            pu[i] = pack_bf16x2(u0, u1);
          }
          store_chunk_coalesced(ph, sbuf, lane, hdst + c, p.out_cols, valid_rows);
          store_chunk_coalesced(pg, sbuf, lane, gdst + c, 2 * p.out_cols, valid_rows);
          store_chunk_coalesced(pu, sbuf, lane, gdst + H + c, 2 * p.out_cols, valid_rows);
        }
      } else if constexpr (M == Mode::kDgradSwiGLU) {
        const int kCols = BN / 2;
        const int c0 = halfc * kCols;
        const int H = p.half;
        const int64_t ld = 2 * static_cast<int64_t>(p.out_cols);  // G,U and dG,dU rows: 2f
#pragma unroll 1
        for (int c = 0; c < kCols; c += 32) {
          // column j of dH is gate column j: interleaved tile j / H, offset j % H
          const int j = nt * BN + c0 + c;
          const int64_t gcol = static_cast<int64_t>(j / H) * 2 * H + j % H;
          uint32_t dh[32];
          tmem_ld_32x32(taddr + c0 + c, dh);
          uint32_t gw[16], uw[16];
          load_chunk_coalesced(gw, sbuf, lane, p.gu + wrow0 * ld + gcol, ld, valid_rows);
          load_chunk_coalesced(uw, sbuf, lane, p.gu + wrow0 * ld + gcol + H, ld, valid_rows);
          tmem_ld_wait();
          if (c + 32 == kCols) release_accumulator();
          uint32_t pdg[16], pdu[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[i]));
            const float2 uf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&uw[i]));
            const float d0 = __uint_as_float(dh[2 * i]), d1 = __uint_as_float(dh[2 * i + 1]);
            const float s0 = sigmoid_f32(gf.x), s1 = sigmoid_f32(gf.y);
            // Silu(g) = g s;  Silu'(g) = s (1 + g (1 - s))
            pdg[i] = pack_bf16x2(d0 * uf.x * s0 * (1.0f + gf.x * (1.0f - s0)),
                                 d1 * uf.y * s1 * (1.0f + gf.y * (1.0f - s1)));
            pdu[i] = pack_bf16x2(d0 * gf.x * s0, d1 * gf.y * s1);
          }
          store_chunk_coalesced(pdg, sbuf, lane, p.out + wrow0 * ld + gcol, ld, valid_rows);
          store_chunk_coalesced(pdu, sbuf, lane, p.out + wrow0 * ld + gcol + H, ld, valid_rows);
        }
      } else {
        const int kCols = BN / 2;
        const int c0 = halfc * kCols;
#pragma unroll 1
        for (int c = 0; c < kCols; c += 32) {
          const int n = nt * BN + c0 + c;
          uint32_t v[32];
          if (k_rows > 0) {
            tmem_ld_32x32(taddr + c0 + c, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;  // an expert without rows: zero gradient
          }
          if (c + 32 == kCols) release_accumulator();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) packed[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          if constexpr (kW) {
            // the 32 x 32 chunk goes out with one TMA store from the staging
            // buffer (rows of 64 bytes, 16-byte pieces permuted by (row >> 1) & 3
            // = the 64-byte swizzle); the previous store has read the buffer.
            // (The gradient's rows come in multiples of 64, so a chunk has all
            // 32 of its rows or none.)
            if (valid_rows == 32) {
              if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
              __syncwarp();
#pragma unroll
              for (int j = 0; j < 4; ++j)
                sbuf[lane * 4 + (j ^ ((lane >> 1) & 3))] =
                    make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
              __syncwarp();
              if (lane == 0) {
                const CUtensorMap* map = &tm_o1;
                int32_t x = n;
                if (p.interleaved) {
                  // interleaved gate/up column n -> gate or up column of [E, d, f]
                  const int H = p.half;
                  const int within = n % (2 * H);
                  x = (n / (2 * H)) * H + within % H;
                  if (within >= H) map = &tm_o2;
                }
                const int32_t y = static_cast<int32_t>(static_cast<int64_t>(e) * p.M_ext + wrow0);
                asm volatile(
                    "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                        reinterpret_cast<uint64_t>(map)),
                    "r"(smem_addr(sbuf)), "r"(x), "r"(y)
                    : "memory");
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
              }
              continue;
            }
            if (valid_rows == 0) continue;
          }
          __nv_bfloat16* dst;
          int64_t ld;
          if constexpr (kW) {
            if (p.interleaved) {
              // interleaved gate/up column n -> gate or up column j of [E, d, f]
              const int H = p.half;
              const int within = n % (2 * H);
              const int jcol = (n / (2 * H)) * H + within % H;
              ld = p.out_cols;
              dst = (within >= H ? p.out2 : p.out) + static_cast<int64_t>(e) * p.M_ext * ld + wrow0 * ld + jcol;
            } else {
              ld = p.N_ext;
              dst = p.out + static_cast<int64_t>(e) * p.M_ext * ld + wrow0 * ld + n;
            }
          } else {
            ld = p.out_cols;
            dst = p.out + wrow0 * ld + n;
          }
          store_chunk_coalesced(packed, sbuf, lane, dst, ld, valid_rows);
        }
      }
      acc ^= 1;
      if (acc == 0) aphase ^= 1u;
    }
    if constexpr (kW)
      if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // the last stores completed
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

int tile_n_for(int n) { return n % 256 == 0 ? 256 : n % 128 == 0 ? 128 : 64; }

template <int BN, Mode M>
cudaError_t launch_mode(const CUtensorMap& ma, const CUtensorMap& mb, const Params& prm, int64_t max_tiles,
                        int num_sms, cudaStream_t stream, const CUtensorMap* mo1 = nullptr,
                        const CUtensorMap* mo2 = nullptr) {
  using C = Cfg<BN, M>;
  const size_t smem = 1024 + static_cast<size_t>(C::kStages) * C::kStageBytes + sizeof(Smem) +
                      2 * static_cast<size_t>(prm.E + 1) * sizeof(int32_t) + 1024 + kStoreStageBytes;
  auto kernel = grouped_gemm_bwd_kernel<BN, M>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const int grid = static_cast<int>(max_tiles < num_sms ? max_tiles : num_sms);
  // output maps: the weight gradients' TMA stores (other modes pass an unused copy)
  kernel<<<grid, kThreads, smem, stream>>>(ma, mb, mo1 ? *mo1 : ma, mo2 ? *mo2 : ma, prm);
  return cudaGetLastError();
}

template <Mode M>
cudaError_t launch_tile_n(int bn, const CUtensorMap& ma, const CUtensorMap& mb, const Params& prm,
                          int64_t max_tiles, int num_sms, cudaStream_t stream, const CUtensorMap* mo1 = nullptr,
                          const CUtensorMap* mo2 = nullptr) {
  switch (bn) {
    case 256: return launch_mode<256, M>(ma, mb, prm, max_tiles, num_sms, stream, mo1, mo2);
    case 128: return launch_mode<128, M>(ma, mb, prm, max_tiles, num_sms, stream, mo1, mo2);
    default: return launch_mode<64, M>(ma, mb, prm, max_tiles, num_sms, stream, mo1, mo2);
  }
}

Params base_params(const int32_t* offsets, int E, int32_t* counter, int32_t* status) {
  Params prm{};
  prm.offsets = offsets;
  prm.E = E;
  prm.tile_counter = counter;
  prm.status = status;
  return prm;
}

}  // namespace

cudaError_t launch_gate_up_save(const BackwardGemmArgs& a, int num_sms, cudaStream_t stream) {
  if (a.P == 0) return cudaSuccess;
  {
    // the forward's paired-SM GEMM writes G and U beside H where it applies
    GroupedGemmProblem g{a.x_perm, a.w_gate_up, a.offsets, nullptr, a.h, a.P, a.E, a.d, 2 * a.f, a.f,
                         a.counters + 0, a.status};
    g.gu_out = a.gu;
    if (grouped_gemm_2sm_supported(g, Epilogue::kSwiGLU)) return launch_grouped_gemm_2sm(g, Epilogue::kSwiGLU, num_sms,
                                                                                           stream);
  }
  const int bn = gate_up_tile_n(a.f);
  CUtensorMap ma, mb;
  if (!make_bf16_map_2d(&ma, a.x_perm, a.P, a.d, BK, BM)) return cudaErrorInvalidValue;
  const int64_t blocks = static_cast<int64_t>(a.E) * (2 * a.f / bn) * (a.d / BK);
  if (!make_bf16_map_3d(&mb, a.w_gate_up, BK, bn, blocks, BK, bn)) return cudaErrorInvalidValue;
  Params prm = base_params(a.offsets, a.E, a.counters + 0, a.status);
  prm.K = a.d;
  prm.n_tiles = 2 * a.f / bn;
  prm.out = static_cast<__nv_bfloat16*>(a.h);
  prm.out2 = static_cast<__nv_bfloat16*>(a.gu);
  prm.out_cols = a.f;
  const int64_t max_tiles = (a.P / BM + a.E) * static_cast<int64_t>(prm.n_tiles);
  return bn == 256 ? launch_mode<256, Mode::kGateUpSave>(ma, mb, prm, max_tiles, num_sms, stream)
                   : launch_mode<128, Mode::kGateUpSave>(ma, mb, prm, max_tiles, num_sms, stream);
}

bool backward_gate_grad_in_dgrad(int E, int d, int f) {
  DgradProblem gd{nullptr, nullptr, nullptr, 0, E, d, f, down_tile_n(d), d / down_tile_n(d),
                  DgradEpilogue::kSwiGLUBwd, nullptr, nullptr, nullptr, nullptr};
  return dgrad_2sm_supported(gd);
}

cudaError_t launch_backward_dgrad_gemms(const BackwardGemmArgs& a, int num_sms, cudaStream_t stream,
                                        void* const* events) {
  auto mark = [&](int i) -> cudaError_t {
    return events && events[i] ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream) : cudaSuccess;
  };
  const auto* wgu = static_cast<const __nv_bfloat16*>(a.w_gate_up);
  const auto* wdn = static_cast<const __nv_bfloat16*>(a.w_down);
  const int bn_gu = gate_up_tile_n(a.f);  // packed gate/up N tile (2h)
  const int bn_dn = down_tile_n(a.d);     // packed down N tile
  const int64_t mt_bound = a.P / BM + a.E;
  cudaError_t err = cudaSuccess;
  // the dgrad GEMMs run on SM pairs (grouped_gemm_2sm.cu) where the output
  // features per expert are a multiple of 256, else on single SMs below
  DgradProblem gd{a.dy_dgrad ? a.dy_dgrad : a.dy, wdn, a.offsets, a.P, a.E, a.d, a.f, bn_dn, a.d / bn_dn,
                  DgradEpilogue::kSwiGLUBwd, a.gu, a.dgu, a.counters + 2, a.status, a.row_w, a.dh_raw};
  DgradProblem gx{a.dgu, wgu, a.offsets, a.P, a.E, 2 * a.f, a.d, bn_gu, 2 * a.f / bn_gu, DgradEpilogue::kRows,
                  nullptr, a.dx_perm, a.counters + 3, a.status};
  const bool gated_dgrad = a.dy_dgrad != nullptr || a.row_w != nullptr || a.dh_raw != nullptr;
  if (gated_dgrad && !dgrad_2sm_supported(gd)) return cudaErrorNotSupported;
  if (a.P > 0 && dgrad_2sm_supported(gd)) {
    if ((err = launch_dgrad_2sm(gd, num_sms, stream)) != cudaSuccess) return err;
  } else if (a.P > 0) {
    // dH = dY Wd^T with dG, dU in the epilogue: N = f, K = d, B from packed down
    {
      const int bn = tile_n_for(a.f);
      CUtensorMap ma, mb;
      if (!make_bf16_map_2d(&ma, a.dy, a.P, a.d, BK, BM)) return cudaErrorInvalidValue;
      const int64_t blocks = static_cast<int64_t>(a.E) * (a.d / bn_dn) * (a.f / BK);
      if (!make_bf16_map_3d(&mb, wdn, BK, bn_dn, blocks, BK, 64, bn / 64)) return cudaErrorInvalidValue;
      Params prm = base_params(a.offsets, a.E, a.counters + 2, a.status);
      prm.K = a.d;
      prm.n_tiles = a.f / bn;
      prm.N_ext = a.f;
      prm.b_rows = bn_dn;
      prm.b_tiles = a.d / bn_dn;
      prm.b_kblocks = a.f / BK;
      prm.half = gate_up_half_tile(a.f);
      prm.gu = static_cast<const __nv_bfloat16*>(a.gu);
      prm.out = static_cast<__nv_bfloat16*>(a.dgu);
      prm.out_cols = a.f;
      err = launch_tile_n<Mode::kDgradSwiGLU>(bn, ma, mb, prm, mt_bound * prm.n_tiles, num_sms, stream);
      if (err != cudaSuccess) return err;
    }
  }
  if ((err = mark(0)) != cudaSuccess) return err;
  if (a.P > 0 && dgrad_2sm_supported(gx)) {
    if ((err = launch_dgrad_2sm(gx, num_sms, stream)) != cudaSuccess) return err;
  } else if (a.P > 0) {
    // dX = [dG | dU] [Wg ; Wu]^T: N = d, K = 2f (interleaved), B from packed gate/up
    {
      const int bn = tile_n_for(a.d);
      CUtensorMap ma, mb;
      if (!make_bf16_map_2d(&ma, a.dgu, a.P, 2 * a.f, BK, BM)) return cudaErrorInvalidValue;
      const int64_t blocks = static_cast<int64_t>(a.E) * (2 * a.f / bn_gu) * (a.d / BK);
      if (!make_bf16_map_3d(&mb, wgu, BK, bn_gu, blocks, BK, 64, bn / 64)) return cudaErrorInvalidValue;
      Params prm = base_params(a.offsets, a.E, a.counters + 3, a.status);
      prm.K = 2 * a.f;
      prm.n_tiles = a.d / bn;
      prm.N_ext = a.d;
      prm.b_rows = bn_gu;
      prm.b_tiles = 2 * a.f / bn_gu;
      prm.b_kblocks = a.d / BK;
      prm.out = static_cast<__nv_bfloat16*>(a.dx_perm);
      prm.out_cols = a.d;
      err = launch_tile_n<Mode::kDgradPlain>(bn, ma, mb, prm, mt_bound * prm.n_tiles, num_sms, stream);
      if (err != cudaSuccess) return err;
    }
  }
  return mark(1);
}

cudaError_t launch_backward_wgrad_gemms(const BackwardGemmArgs& a, int num_sms, cudaStream_t stream,
                                        void* const* events) {
  auto mark = [&](int i) -> cudaError_t {
    return events && events[i] ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream) : cudaSuccess;
  };
  cudaError_t err = cudaSuccess;
  const void* h_w = a.h_wgrad ? a.h_wgrad : a.h;
  const void* dy_w = a.dy_wgrad ? a.dy_wgrad : a.dy;
  // dWd[e] = H_e^T dY_e: M = f, N = d, K = the expert's rows
  if (a.dw_down) {
    const int bn = tile_n_for(a.d);
    CUtensorMap ma, mb;
    const int64_t rows = a.P > 0 ? a.P : 1;
    if (!make_bf16_map_col_blocks(&ma, a.P > 0 ? h_w : a.dw_down, rows, a.f, BK, BM / 64)) return cudaErrorInvalidValue;
    if (!make_bf16_map_col_blocks(&mb, a.P > 0 ? dy_w : a.dw_down, rows, a.d, BK, bn / 64)) return cudaErrorInvalidValue;
    Params prm = base_params(a.offsets, a.E, a.counters + 4, a.status);
    prm.m_tiles = (a.f + BM - 1) / BM;
    prm.n_tiles = a.d / bn;
    prm.M_ext = a.f;
    prm.N_ext = a.d;
    prm.out = static_cast<__nv_bfloat16*>(a.dw_down);
    CUtensorMap mo;  // dW_down [E * f, d]: 32 x 32 store boxes
    if (!make_bf16_map_2d_sw64(&mo, a.dw_down, static_cast<int64_t>(a.E) * a.f, a.d, 32, 32))
      return cudaErrorInvalidValue;
    err = launch_tile_n<Mode::kWgrad>(bn, ma, mb, prm, static_cast<int64_t>(a.E) * prm.m_tiles * prm.n_tiles, num_sms,
                                      stream, &mo, &mo);
    if (err != cudaSuccess) return err;
  }
  if ((err = mark(0)) != cudaSuccess) return err;
  // dWg[e] = X_e^T dG_e, dWu[e] = X_e^T dU_e: M = d, N = 2f interleaved
  if (a.dw_gate) {
    const int bn = tile_n_for(2 * a.f);  // may span two interleaved gate/up tiles
    CUtensorMap ma, mb;
    const int64_t rows = a.P > 0 ? a.P : 1;
    if (!make_bf16_map_col_blocks(&ma, a.P > 0 ? a.x_perm : a.dw_gate, rows, a.d, BK, BM / 64))
      return cudaErrorInvalidValue;
    if (!make_bf16_map_col_blocks(&mb, a.P > 0 ? a.dgu : a.dw_gate, rows, 2 * a.f, BK, bn / 64))
      return cudaErrorInvalidValue;
    Params prm = base_params(a.offsets, a.E, a.counters + 5, a.status);
    prm.m_tiles = (a.d + BM - 1) / BM;
    prm.n_tiles = 2 * a.f / bn;
    prm.M_ext = a.d;
    prm.N_ext = 2 * a.f;
    prm.half = gate_up_half_tile(a.f);
    prm.interleaved = 1;
    prm.out = static_cast<__nv_bfloat16*>(a.dw_gate);
    prm.out2 = static_cast<__nv_bfloat16*>(a.dw_up);
    prm.out_cols = a.f;
    CUtensorMap mg, mu;  // dW_gate, dW_up [E * d, f]: 32 x 32 store boxes
    if (!make_bf16_map_2d_sw64(&mg, a.dw_gate, static_cast<int64_t>(a.E) * a.d, a.f, 32, 32) ||
        !make_bf16_map_2d_sw64(&mu, a.dw_up, static_cast<int64_t>(a.E) * a.d, a.f, 32, 32))
      return cudaErrorInvalidValue;
    err = launch_tile_n<Mode::kWgrad>(bn, ma, mb, prm, static_cast<int64_t>(a.E) * prm.m_tiles * prm.n_tiles, num_sms,
                                      stream, &mg, &mu);
    if (err != cudaSuccess) return err;
  }
  return mark(1);
}

cudaError_t launch_swiglu_backward_gemms(const BackwardGemmArgs& a, int num_sms, cudaStream_t stream,
                                         void* const* events) {
  cudaError_t err = launch_backward_dgrad_gemms(a, num_sms, stream, events);
  if (err != cudaSuccess) return err;
  return launch_backward_wgrad_gemms(a, num_sms, stream, events ? events + 2 : nullptr);
}

}  // namespace moe
