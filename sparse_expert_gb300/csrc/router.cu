// Router linear layer fused with Softmax and TopK ("Scalable Pretraining of
// Large MoE LMs on Aurora Super Computer", §3.1, Algorithm 1, stage 1:
// logits = Router(input); probs = Softmax(logits); TopK(probs)).
//
// One block per 128-token tile.  The logits of the tile, 128 x E_pad fp32,
// are accumulated by tcgen05 MMAs (M=128, N=256 or 128, K=16) in tensor
// memory from TMA-fed bf16 tiles of x and of the packed router weights, and
// never reach global memory: the epilogue gives each thread one token row,
// which it reads 32 columns at a time and reduces to its k best experts
// (64-bit (logit, expert) keys, same order and ties as moe_route_topk) and,
// without renormalisation, to an online softmax denominator over all E.
//
// Packed router weights: K-major, [d/64][E_pad][64] bf16 (E padded with
// zero columns to a multiple of 128, E_pad <= 512), so one K block of all
// experts is one contiguous block.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

int router_e_pad(int E) { return (E + 127) / 128 * 128; }

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kABytes = BM * BK * 2;
constexpr int kSmemBudget = 227 * 1024 - 2048 - 4096;  // stages; slack, barriers and the histogram

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
__global__ void __launch_bounds__(kThreads, 1)
router_topk_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                   const RouterParams p) {
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const int b_bytes = p.E_pad * BK * 2;
  const int stage_bytes = kABytes + b_bytes;
  const int stages = min(8, kSmemBudget / stage_bytes);
  __shared__ uint64_t full[8], empty[8], tfull;
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &abort_flag_s;
  const int tmem_cols = p.E_pad <= 128 ? 128 : p.E_pad <= 256 ? 256 : 512;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * BM;
  const int num_kb = p.K / BK;

  if (warp == 1) {
    tmem_alloc(&tmem_base_slot, tmem_cols);
    tmem_relinquish();
  } else if (warp == 0 && lane == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&tfull, 1);
    abort_flag_s = 0;
    fence_barrier_init();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = tmem_base_slot;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_w);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int last_stage = -1;
      uint32_t last_phase = 0;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* sa = base + stage * stage_bytes;
        uint8_t* sb = sa + kABytes;
        mbar_arrive_expect_tx(&full[stage], stage_bytes);
        tma_load_2d(sa, &tm_x, &full[stage], kb * BK, static_cast<int32_t>(m0));
        for (int c = 0; c < p.E_pad; c += 128) tma_load_3d(sb + c * BK * 2, &tm_w, &full[stage], 0, c, kb);
        last_stage = stage;
        last_phase = phase;
        if (++stage == stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        record_status(p.status, kStatusTimeout);
        *abort_flag = 1;
        if (last_stage >= 0) {
          volatile int never = 0;
          mbar_wait(&full[last_stage], last_phase, &never);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a0 = smem_addr(base + stage * stage_bytes);
        const uint32_t b0 = a0 + kABytes;
#pragma unroll
        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
          const uint64_t da = sw128_kmajor_desc(a0 + kk * UMMA_K * 2);
          for (int n0 = 0; n0 < p.E_pad; n0 += 256) {
            const int n = min(256, p.E_pad - n0);
            const uint32_t idesc = n == 256 ? umma_idesc_bf16_f32(BM, 256) : umma_idesc_bf16_f32(BM, 128);
            umma_bf16(tmem_base + n0, da, sw128_kmajor_desc(b0 + n0 * BK * 2 + kk * UMMA_K * 2), idesc,
                      (kb | kk) != 0 ? 1u : 0u);
          }
        }
        umma_commit(&empty[stage]);
        if (++stage == stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        record_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      umma_commit(&tfull);  // also completes once every issued MMA is done
    }
  } else {
    // ---- epilogue: thread = token row
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int64_t t = m0 + row;
    const bool valid = t < p.T;
    const bool done = mbar_wait_warp(&tfull, 0, abort_flag);
    if (!done && lane == 0) {
      record_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    if (done) {
      tc_fence_after_sync();
      uint64_t best[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) best[j] = 0;
      float run_max = -INFINITY, run_sum = 0.f;  // online softmax over all E (no renormalisation)
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
      for (int c0 = 0; c0 < p.E_pad; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32x32(taddr + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c0 + i;
          if (e >= p.E) break;
          const float x = __uint_as_float(v[i]);
          uint64_t key = route_key(x, e);
          if (key > best[KMAX - 1]) {
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
              if (key > best[j]) {
                const uint64_t tmp = best[j];
                best[j] = key;
                key = tmp;
              }
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
      const float mx = key_logit(best[0]);
      float denom = run_sum;  // run_max == mx
      if (p.renormalize) {
        denom = 0.f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < p.k) denom += expf(key_logit(best[j]) - mx);
      }
      if (valid) {
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

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, tmem_cols);
  }
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
  const int stage_bytes = kABytes + router_e_pad(E) * BK * 2;
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
  // packed router weights as [d/64][E_pad rows][64], box 128 rows of one block
  if (!make_bf16_map_3d(&mw, w_packed, BK, e_pad, d / BK, BK, 128)) return cudaErrorInvalidValue;
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
  const unsigned grid = static_cast<unsigned>((T + BM - 1) / BM);
  cudaError_t err;
  if (k <= 2) {
    err = cudaFuncSetAttribute(router_topk_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err == cudaSuccess) router_topk_kernel<2><<<grid, kThreads, smem, stream>>>(mx, mw, prm);
  } else if (k <= 8) {
    err = cudaFuncSetAttribute(router_topk_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err == cudaSuccess) router_topk_kernel<8><<<grid, kThreads, smem, stream>>>(mx, mw, prm);
  } else {
    err = cudaFuncSetAttribute(router_topk_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err == cudaSuccess) router_topk_kernel<32><<<grid, kThreads, smem, stream>>>(mx, mw, prm);
  }
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace moe
