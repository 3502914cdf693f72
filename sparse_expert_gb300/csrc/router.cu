// Router linear layer fused with Softmax and TopK ("Scalable Pretraining of
// Large MoE LMs on Aurora Super Computer", §3.1, Algorithm 1, stage 1:
// logits = Router(input); probs = Softmax(logits); TopK(probs)).
//
// One SM pair (a 2-CTA cluster, tcgen05 cta_group::2) per 256-token tile:
// CTA r holds tokens 128r .. 128r+127 of the tile and, of each MMA's expert
// columns, its half, so each SM streams half of the router weights per K
// block instead of all of them.  The leader issues M = 256 MMAs (N = 256 or
// 128 expert columns, K = 16) from TMA-fed bf16 tiles; each CTA's tensor
// memory receives its 128 tokens x E_pad fp32 logits, which never reach
// global memory: the epilogue gives each thread one token row, which it
// reads 32 columns at a time and reduces to its k best experts (64-bit
// (logit, expert) keys, same order and ties as moe_route_topk) and, without
// renormalisation, to an online softmax denominator over all E.
//
// Packed router weights: K-major, [d/64][E_pad][64] bf16 (E padded with
// zero columns to a multiple of 128, E_pad <= 512), so one K block of all
// experts is one contiguous block.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "pair_common.cuh"

namespace moe {

int router_e_pad(int E) { return (E + 127) / 128 * 128; }

namespace {

constexpr int BM = 128;          // token rows per CTA (256 per pair)
constexpr int BK = 64;
constexpr int UMMA_K = 16;
// Warps: 0 TMA, 1 MMA (leader), then kSlices epilogue warps per TMEM lane
// quadrant: each token's expert columns are split into kSlices slices, one
// per warp, whose top-k lists are merged at the end (a thread alone walking
// all E columns of its token spends most of its time in the insertion path,
// because some lane of its warp inserts at nearly every column).
template <int KMAX>
struct RouterCfg {
  static constexpr int kSlices = KMAX <= 8 ? 4 : 2;
  static constexpr int kEpiThreads = 128 * kSlices;
  static constexpr int kThreads = 64 + kEpiThreads;
};
constexpr int kABytes = BM * BK * 2;
constexpr int kBoxRows = 64;     // router-weight rows per TMA box
constexpr int kSmemBudget = 227 * 1024 - 2048 - 4096;  // stages; slack, barriers and the histogram


// One stage of a CTA: its 128 token rows and its half of every MMA's expert
// rows (E_pad / 2 rows) for one K block.
__host__ __device__ constexpr int router_stage_bytes(int e_pad) { return kABytes + (e_pad / 2) * BK * 2; }

struct RouterParams {
  int64_t T;
  int E, E_pad, K, k, renormalize;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* hist;   // per-chunk count table [pairs / 2048][E4], or null
  int E4;
  int32_t* status;
};

__device__ __forceinline__ uint64_t route_key(float x, int e) {
  uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(e));
}

__device__ __forceinline__ float key_logit(uint64_t key) {
  uint32_t u = static_cast<uint32_t>(key >> 32);
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(u);
}

template <int KMAX>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(RouterCfg<KMAX>::kThreads, 1)
router_topk_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                   const RouterParams p) {
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const int stage_bytes = router_stage_bytes(p.E_pad);
  const int stages = min(8, kSmemBudget / stage_bytes);
  __shared__ uint64_t full[8], empty[8], tfull;
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  volatile int* abort_flag = &abort_flag_s;
  const int tmem_cols = p.E_pad <= 128 ? 128 : p.E_pad <= 256 ? 256 : 512;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x >> 1) * (2 * BM) + static_cast<int64_t>(rank) * BM;
  const int num_kb = p.K / BK;
  bool failed = false;

  if (warp == 1) {
    tmem_alloc_pair(&tmem_base_slot, tmem_cols);
  } else if (warp == 0 && lane == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&full[i], 1);   // the leader's producer: both CTAs' bytes
      mbar_init(&empty[i], 1);  // the leader's MMA commit, multicast to both CTAs
    }
    mbar_init(&tfull, 1);
    abort_flag_s = 0;
    fence_barrier_init();
  }
  tc_fence_before_sync();
  cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = tmem_base_slot;

  if (warp == 0) {
    // ---- TMA producer (both CTAs): its 128 token rows and, of each MMA's
    // n expert rows n0 .. n0+n-1, rows n0 + rank*n/2 .. +n/2, stored from
    // row n0/2 of its B stage; every copy counts on the leader's barrier
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_w);
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
          failed = true;
          break;
        }
        uint8_t* sa = base + stage * stage_bytes;
        uint8_t* sb = sa + kABytes;
        const uint32_t lead_full = leader_addr(&full[stage]);
        if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * stage_bytes);
        tma_load_2d_pair(sa, &tm_x, lead_full, kb * BK, static_cast<int32_t>(m0));
        for (int n0 = 0; n0 < p.E_pad; n0 += 256) {
          const int half = min(256, p.E_pad - n0) / 2;
          for (int r = 0; r < half; r += kBoxRows)
            tma_load_3d_pair(sb + (n0 / 2 + r) * BK * 2, &tm_w, lead_full, 0,
                             n0 + static_cast<int>(rank) * half + r, kb);
        }
        if (++stage == stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer (leader): M = 256 tokens of the pair
    if (rank == 0 && lane == 0) {
      // at most two MMAs per K step: expert columns 0 .. n0-1 and n0 .. E_pad-1
      const bool two_parts = p.E_pad > 256;
      const uint32_t idesc0 = umma_idesc_bf16_f32(2 * BM, min(256, p.E_pad));
      const uint32_t idesc1 = umma_idesc_bf16_f32(2 * BM, two_parts ? p.E_pad - 256 : 16);
      const uint64_t b1_off = (128 * BK * 2) >> 4;  // the second part's half starts at B row 128
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag)) {
          failed = true;
          break;
        }
        tc_fence_after_sync();
        // descriptors of the stage's operands; a K step of 16 advances the
        // start-address field (16-byte units) by 2
        const uint64_t da = sw128_kmajor_desc(smem_addr(base + stage * stage_bytes));
        const uint64_t db = sw128_kmajor_desc(smem_addr(base + stage * stage_bytes + kABytes));
#pragma unroll
        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
          const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
          umma_pair(tmem_base, da + 2 * kk, db + 2 * kk, idesc0, acc);
          if (two_parts) umma_pair(tmem_base + 256, da + 2 * kk, db + b1_off + 2 * kk, idesc1, acc);
        }
        umma_commit_pair(&empty[stage]);
        if (++stage == stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      umma_commit_pair(&tfull);  // also completes once every issued MMA is done
    }
  } else {
    // ---- epilogue: thread = token row x one slice of the expert columns
    using RC = RouterCfg<KMAX>;
    const int quad = warp & 3;
    const int slice = (warp - 2) >> 2;
    const int row = quad * 32 + lane;
    const int64_t t = m0 + row;
    const int cols = p.E_pad / RC::kSlices;  // a multiple of 32
    // the merge's scratch: the stage buffers, free once every MMA is done;
    // keys [slice][j][row] and (max, sum) [slice][row], both row-contiguous
    uint64_t* s_keys = reinterpret_cast<uint64_t*>(base);
    float2* s_stat = reinterpret_cast<float2*>(s_keys + RC::kSlices * KMAX * BM);
    const bool done = mbar_wait_warp_suspend(&tfull, 0, abort_flag);
    if (!done) {
      failed = true;
      if (lane == 0) *abort_flag = 1;
    } else {
      tc_fence_after_sync();
      // the slice's k best as logits and experts, best first; experts come in
      // increasing order, so a strictly greater logit is needed to enter, and
      // an equal logit seen earlier (a smaller expert) keeps its place -- the
      // order of the 64-bit keys of moe_route_topk
      float bl[KMAX];
      int be[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        bl[j] = -INFINITY;
        be[j] = 0;
      }
      float run_max = -INFINITY, run_sum = 0.f;  // online softmax over the slice (no renormalisation)
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
      for (int c0 = slice * cols; c0 < (slice + 1) * cols; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32x32(taddr + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c0 + i;
          if (e >= p.E) break;
          const float x = __uint_as_float(v[i]);
          if (x > bl[KMAX - 1]) {
            // every slot from the old list at once: slot j takes the old
            // j-1 if x beats it, else x if x beats the old j
            bool gt[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j) gt[j] = x > bl[j];
#pragma unroll
            for (int j = KMAX - 1; j > 0; --j) {
              bl[j] = gt[j - 1] ? bl[j - 1] : (gt[j] ? x : bl[j]);
              be[j] = gt[j - 1] ? be[j - 1] : (gt[j] ? e : be[j]);
            }
            if (gt[0]) {
              bl[0] = x;
              be[0] = e;
            }
          }
          if (!p.renormalize) {
            if (x > run_max) {
              run_sum = run_sum * expf(run_max - x) + 1.0f;
              run_max = x;
            } else {
              run_sum += expf(x - run_max);
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        s_keys[(slice * KMAX + j) * BM + row] = bl[j] == -INFINITY ? 0 : route_key(bl[j], be[j]);
      s_stat[slice * BM + row] = make_float2(run_max, run_sum);
    }
    // all epilogue warps, whether or not their wait succeeded
    asm volatile("bar.sync 1, %0;" ::"r"(RC::kEpiThreads) : "memory");
    if (slice == 0 && done && *abort_flag == 0) {
      // merge the slices' sorted lists (keys are distinct: they hold the expert)
      int head[RC::kSlices];
#pragma unroll
      for (int q = 0; q < RC::kSlices; ++q) head[q] = 0;
      uint64_t best[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        uint64_t top = 0;
        int from = 0;
#pragma unroll
        for (int q = 0; q < RC::kSlices; ++q) {
          const uint64_t h = head[q] < KMAX ? s_keys[(q * KMAX + head[q]) * BM + row] : 0;
          if (h > top) {
            top = h;
            from = q;
          }
        }
        best[j] = top;
#pragma unroll
        for (int q = 0; q < RC::kSlices; ++q) head[q] += (q == from) ? 1 : 0;
      }
      const float mx = key_logit(best[0]);
      float denom = 0.f;
      if (p.renormalize) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < p.k) denom += expf(key_logit(best[j]) - mx);
      } else {
        // the slices' online sums rescaled to the overall maximum
#pragma unroll
        for (int q = 0; q < RC::kSlices; ++q) {
          const float2 st = s_stat[q * BM + row];
          if (st.y > 0.f) denom += st.y * expf(st.x - mx);
        }
      }
      if (t < p.T) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (j < p.k) {
            const int e = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best[j]));
            const int64_t pr = t * p.k + j;
            p.topk_idx[pr] = e;
            p.topk_w[pr] = expf(key_logit(best[j]) - mx) / denom;
            if (p.hist) atomicAdd(p.hist + (pr / kDispatchChunk) * p.E4 + e, 1);
          }
        }
      }
    }
  }

  if (failed && lane == 0) {
    record_status(p.status, kStatusTimeout);
    *abort_flag = 1;
  }
  __syncthreads();
  // after a timeout, let copies still in flight land before the pair meets
  // and frees its tensor memory
  if (*abort_flag) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 10000000ull) __nanosleep(1000);
  }
  tc_fence_before_sync();
  cluster_sync();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc_pair(tmem_base, tmem_cols);
}

// packed[((i / 64) * E_pad + e) * 64 + i % 64] = w[i][e] (0 for e >= E)
__global__ void pack_router_kernel(const __nv_bfloat16* __restrict__ w, int d, int E, int E_pad,
                                   __nv_bfloat16* __restrict__ packed) {
  const int64_t n = static_cast<int64_t>(d) * E_pad;
  for (int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; o < n;
       o += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int kk = static_cast<int>(o % 64);
    const int64_t r = o / 64;
    const int e = static_cast<int>(r % E_pad);
    const int i = static_cast<int>(r / E_pad) * 64 + kk;
    packed[o] = e < E ? w[static_cast<int64_t>(i) * E + e] : __float2bfloat16(0.0f);
  }
}

}  // namespace

cudaError_t launch_pack_router(const void* w_router, int d, int E, void* packed, cudaStream_t stream) {
  const int e_pad = router_e_pad(E);
  const int64_t n = static_cast<int64_t>(d) * e_pad;
  const int grid = static_cast<int>((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  pack_router_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(w_router), d, E, e_pad,
                                               static_cast<__nv_bfloat16*>(packed));
  return cudaGetLastError();
}

size_t router_smem_bytes(int E) {
  const int stage_bytes = router_stage_bytes(router_e_pad(E));
  const int stages = kSmemBudget / stage_bytes < 8 ? kSmemBudget / stage_bytes : 8;
  return 1024 + static_cast<size_t>(stages) * stage_bytes + static_cast<size_t>(E) * 4;
}

cudaError_t launch_router_topk(const void* x, const void* w_packed, int64_t T, int d, int E, int k, int renormalize,
                               int32_t* topk_idx, float* topk_w, int32_t* hist, int32_t* status,
                               cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int e_pad = router_e_pad(E);
  CUtensorMap mx, mw;
  if (!make_bf16_map_2d(&mx, x, T, d, BK, BM)) return cudaErrorInvalidValue;
  // packed router weights as [d/64][E_pad rows][64], boxes of 64 rows of one block
  if (!make_bf16_map_3d(&mw, w_packed, BK, e_pad, d / BK, BK, kBoxRows)) return cudaErrorInvalidValue;
  RouterParams prm;
  prm.T = T;
  prm.E = E;
  prm.E_pad = e_pad;
  prm.K = d;
  prm.k = k;
  prm.renormalize = renormalize;
  prm.topk_idx = topk_idx;
  prm.topk_w = topk_w;
  prm.hist = hist;
  prm.E4 = dispatch_hist_stride(E);
  prm.status = status;
  const size_t smem = router_smem_bytes(E);
  const unsigned grid = 2u * static_cast<unsigned>((T + 2 * BM - 1) / (2 * BM));  // one pair per 256 tokens
  cudaError_t err;
  if (k <= 2) {
    err = cudaFuncSetAttribute(router_topk_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err == cudaSuccess) router_topk_kernel<2><<<grid, RouterCfg<2>::kThreads, smem, stream>>>(mx, mw, prm);
  } else if (k <= 8) {
    err = cudaFuncSetAttribute(router_topk_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err == cudaSuccess) router_topk_kernel<8><<<grid, RouterCfg<8>::kThreads, smem, stream>>>(mx, mw, prm);
  } else {
    err = cudaFuncSetAttribute(router_topk_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err == cudaSuccess) router_topk_kernel<32><<<grid, RouterCfg<32>::kThreads, smem, stream>>>(mx, mw, prm);
  }
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace moe
