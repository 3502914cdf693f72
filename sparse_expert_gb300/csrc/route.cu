// Stage 1 of the layer: Softmax and TopK of the router logits, one warp per
// token ("Scalable Pretraining of Large MoE LMs on Aurora Super Computer",
// §3.1, Algorithm 1, stage 1).  Optionally adds each selection to the
// per-chunk count table of stage 2 (one atomic add per pair into
// hist[pair / 2048][expert]) so that the index pass starts from complete
// counts without another read of the indices.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;  // tokens per block

// (logit, expert) as one 64-bit key whose unsigned order is the selection
// order: larger logit first, then the smaller expert index.  The high word
// is the float's bits made monotone (negative values inverted, sign bit set
// on the others) after folding -0.0 onto +0.0 (x + 0.0f: -0.0 + 0.0 is +0.0
// under round to nearest, and every other finite x is unchanged); the low
// word decreases with the expert index.  Key 0 is below every finite
// logit's key.
__device__ __forceinline__ uint32_t route_hi(float x) {
  const uint32_t u = __float_as_uint(__fadd_rn(x, 0.0f));
  const uint32_t neg = static_cast<uint32_t>(static_cast<int32_t>(u) >> 31);  // all ones when negative
  return u ^ (neg | 0x80000000u);
}

__device__ __forceinline__ uint64_t route_key_hi(uint32_t hi, int e) {
  return (static_cast<uint64_t>(hi) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(e));
}

__device__ __forceinline__ uint64_t route_key(float x, int e) { return route_key_hi(route_hi(x), e); }

__device__ __forceinline__ float key_logit(uint64_t key) {
  uint32_t u = static_cast<uint32_t>(key >> 32);
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(u);
}

__device__ __forceinline__ int key_expert(uint64_t key) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key));
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t b) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xffffffffu, b, s);
    b = o > b ? o : b;
  }
  return b;
}

// Bitonic sort of one key per lane over each aligned group of W lanes.
// Lanes 0 .. W-1 end in descending order (the other groups alternate in
// direction, as the network leaves them before a wider merge).
template <int W, typename Key>
__device__ __forceinline__ Key warp_sort_desc(Key v, int lane) {
#pragma unroll
  for (int size = 2; size <= W; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const Key o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      v = keep_max ? (o > v ? o : v) : (o < v ? o : v);
    }
  }
  return v;
}

// Exact top-k of one token's keys by k rounds of warp arg-max: round j takes
// the warp maximum of the lanes' best keys, and only the lane that held it
// marks that key taken and rescans its own values.  Keys are rebuilt from
// the logits on each scan (a taken bit per value instead of a held key), so
// this rarely taken path costs no registers across the common one.  Lane
// j < k gets the j-th key.
template <int NV>
__device__ __forceinline__ uint64_t lane_best_key(const float (&v)[NV], int E, int lane, uint32_t taken) {
  uint64_t b = 0;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    if (e < E && !((taken >> i) & 1u)) {
      const uint64_t key = route_key(v[i], e);
      b = key > b ? key : b;
    }
  }
  return b;
}

template <int NV>
__device__ __forceinline__ uint64_t topk_rounds(const float (&v)[NV], int E, int k, int lane) {
  uint32_t taken = 0;
  uint64_t lbest = lane_best_key<NV>(v, E, lane, taken);
  uint64_t mine = 0;
  for (int j = 0; j < k; ++j) {
    const uint64_t b = warp_max_u64(lbest);
    if (lane == j) mine = b;
    if (lbest == b) {  // keys are unique: exactly one lane held it
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        if (e < E && route_key(v[i], e) == b) taken |= 1u << i;
      }
      lbest = lane_best_key<NV>(v, E, lane, taken);
    }
  }
  return mine;
}

// NV logits per lane: lane l holds experts l, l+32, ..., l+32*(NV-1); with
// kFull every lane holds exactly NV (E = 32 NV) and no index is tested.
//
// Without groups the selection first narrows the field.  Let H be the k-th
// largest of the 32 lanes' maximum logits, or, for k <= 16, the k-th
// largest of the 16 maxima of lane pairs (l, l + 16).  Either way at least k
// distinct experts have a logit >= H, so an expert below H has at least k
// keys above it and cannot be selected: every selected expert is among the
// candidates (logit >= H as a float compare, where -0.0 equals +0.0 exactly
// as in the key order).  A lane without experts contributes -inf, which
// makes every expert a candidate.  For N(0,1) logits over 384 experts there
// are about nine candidates.  When they number at most 32 each is written
// once into the warp's shared buffer and ranked by counting the candidate
// keys above it, and the k of rank < k land in slot order.  Otherwise (wide
// ties) the k rounds of topk_rounds decide.  Both give the k largest keys in
// descending order, so the result does not depend on the path taken.
//
// With n_groups > 1 ("Training a 1T-Params MoE on EU public
// infrastructure", Group-limited expert routing), group g = experts
// [g*E/G, (g+1)*E/G) gets k/G rounds restricted to its own experts, and a
// warp sort puts the k winners back in descending slot order.
//
// The loads of a warp's next token are issued before the current token's
// selection, so their latency overlaps it.
template <int NV, bool kFull, bool kGrouped>
__global__ void __launch_bounds__(kRouteWarps * 32, NV <= 12 ? 4 : NV <= 16 ? 2 : 1)
route_topk_kernel(const float* __restrict__ logits, int64_t T, int E, int k, int n_groups, int renormalize,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ hist, int E4) {
  __shared__ uint64_t s_cand[kRouteWarps * 32];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint64_t* cand = s_cand + warp * 32;

  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * kRouteWarps;
  int64_t t = static_cast<int64_t>(blockIdx.x) * kRouteWarps + warp;
  float v[NV];
  if (!kGrouped && t < T) {
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      v[i] = (kFull || e < E) ? __ldg(logits + t * E + e) : 0.0f;
    }
  }
  for (; t < T; t += warps_total) {
    const int64_t tn = t + warps_total;
    float vn[NV];
    if (kGrouped) {
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        v[i] = (e < E) ? __ldg(logits + t * E + e) : 0.0f;
      }
    } else if (tn < T) {
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        vn[i] = (kFull || e < E) ? __ldg(logits + tn * E + e) : 0.0f;
      }
    }
    uint64_t mine = 0, first = 0;
    if (!kGrouped) {
      float hm = -INFINITY;
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (kFull || lane + 32 * i < E) hm = fmaxf(hm, v[i]);
      float H;  // the same in every lane
      if (k <= 16) {
        const float hp = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 16));
        H = __shfl_sync(0xffffffffu, warp_sort_desc<16>(hp, lane), k - 1);
      } else {
        H = __shfl_sync(0xffffffffu, warp_sort_desc<32>(hm, lane), k - 1);
      }
      // candidates column by column: one ballot per column, skipped by the
      // whole warp when the column holds none; the buffer takes the first
      // 32 in (column, lane) order and C counts them all
      const unsigned lanes_below = (1u << lane) - 1u;
      uint32_t C = 0;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        const bool is_cand = (kFull || e < E) && v[i] >= H;
        const unsigned mask = __ballot_sync(0xffffffffu, is_cand);
        if (mask) {
          const uint32_t pos = C + __popc(mask & lanes_below);
          if (is_cand && pos < 32) cand[pos] = route_key(v[i], e);
          C += __popc(mask);
        }
      }
      if (C <= 32) {
        __syncwarp();
        const uint64_t c = (static_cast<uint32_t>(lane) < C) ? cand[lane] : 0ull;
        uint32_t rank = 0;
#pragma unroll 4
        for (uint32_t j = 0; j < C; ++j) rank += cand[j] > c ? 1u : 0u;
        __syncwarp();
        if (static_cast<uint32_t>(lane) < C && rank < static_cast<uint32_t>(k)) cand[rank] = c;
        __syncwarp();
        mine = (lane < k) ? cand[lane] : 0ull;
        __syncwarp();
      } else {
        mine = topk_rounds<NV>(v, E, k, lane);
      }
      first = __shfl_sync(0xffffffffu, mine, 0);
    } else {
      uint64_t key[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        key[i] = (e < E) ? route_key(v[i], e) : 0ull;
      }
      const int gsize = E / n_groups, per = k / n_groups;
      int j = 0;
      for (int g = 0; g < n_groups; ++g) {
        const int lo = g * gsize, hi = lo + gsize;
        for (int r = 0; r < per; ++r, ++j) {
          uint64_t lb = 0;
#pragma unroll
          for (int i = 0; i < NV; ++i) {
            const int e = lane + 32 * i;
            if (e >= lo && e < hi && key[i] > lb) lb = key[i];
          }
          const uint64_t b = warp_max_u64(lb);
          if (lane == j) mine = b;
#pragma unroll
          for (int i = 0; i < NV; ++i)
            if (key[i] == b) key[i] = 0;
        }
      }
      mine = warp_sort_desc<32>(mine, lane);  // lanes >= k hold key 0
      first = __shfl_sync(0xffffffffu, mine, 0);
    }
    const float mx = key_logit(first);
    const float z = (lane < k) ? expf(key_logit(mine) - mx) : 0.0f;
    float denom = 0.0f;
    if (renormalize) {
      denom = z;
    } else {
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (lane + 32 * i < E) denom += expf(v[i] - mx);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, s);
    denom = __shfl_sync(0xffffffffu, denom, 0);  // one rounding for every slot
    if (lane < k) {
      const int e = key_expert(mine);
      const int64_t p = t * k + lane;
      topk_idx[p] = e;
      topk_w[p] = z / denom;
      if (hist) atomicAdd(hist + (p / kDispatchChunk) * E4 + e, 1);
    }
    if (!kGrouped) {
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] = vn[i];
    }
  }
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, int64_t T, int E, int k, int n_groups, int renormalize,
                              int32_t* topk_idx, float* topk_w, int32_t* hist, int num_sms, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int64_t blocks_needed = (T + kRouteWarps - 1) / kRouteWarps;
  const int64_t max_blocks = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(blocks_needed < max_blocks ? blocks_needed : max_blocks);
  const int E4 = dispatch_hist_stride(E);
  const int nv = (E + 31) / 32;
#define MOE_ROUTE_LAUNCH(NV, FULL, GROUPED)                                                               \
  route_topk_kernel<NV, FULL, GROUPED><<<grid, kRouteWarps * 32, 0, stream>>>(logits, T, E, k, n_groups,      \
                                                                               renormalize, topk_idx, topk_w, \
                                                                               hist, E4)
#define MOE_ROUTE_CASE(NV)                               \
  if (n_groups > 1)                                      \
    MOE_ROUTE_LAUNCH(NV, false, true);                   \
  else if (E == 32 * (NV))                               \
    MOE_ROUTE_LAUNCH(NV, true, false);                   \
  else                                                   \
    MOE_ROUTE_LAUNCH(NV, false, false);                  \
  break;
  switch (nv <= 1 ? 1 : nv <= 2 ? 2 : nv <= 4 ? 4 : nv <= 8 ? 8 : nv <= 12 ? 12 : nv <= 16 ? 16 : 32) {
    case 1: MOE_ROUTE_CASE(1)
    case 2: MOE_ROUTE_CASE(2)
    case 4: MOE_ROUTE_CASE(4)
    case 8: MOE_ROUTE_CASE(8)
    case 12: MOE_ROUTE_CASE(12)
    case 16: MOE_ROUTE_CASE(16)
    default: MOE_ROUTE_CASE(32)
  }
#undef MOE_ROUTE_LAUNCH
#undef MOE_ROUTE_CASE
  return cudaGetLastError();
}

}  // namespace moe
