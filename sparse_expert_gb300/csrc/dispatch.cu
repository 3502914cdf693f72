// Stages 2 and 3 of the layer: per-expert token counts, their prefix sums,
// and the index maps ("Scalable Pretraining of Large MoE LMs on Aurora
// Super Computer", §3.1, Algorithm 1, stages 2-3).
//
// The page's kernels give each thread a block of tokens, count per
// (expert, thread), prefix-sum the expert-major count table, and let each
// (expert, thread) write rows from its base with a running counter.  The
// result is a stable counting sort of the pairs by expert.  Here the same
// sort is done by blocks of 2,048 consecutive pairs:
//   1. a histogram gives complete per-expert counts (or the route kernel
//      produces them on the fly);
//   2. one pass in which every block ranks its pairs within the block
//      (warp match + per-warp running counts), publishes its per-expert
//      aggregate, and takes the exclusive per-expert prefix of all earlier
//      blocks by decoupled look-back (Merrill & Garland's single-pass scan,
//      applied to an E-wide vector, with the predecessors' flags read 32 at
//      a time so that the walk costs one round trip per 32 blocks).  Block
//      order comes from an atomic ticket, so a block only ever waits for
//      blocks that are already running, and every wait is bounded.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kWarps = kDispatchThreads / 32;
constexpr int32_t kFlagAggregate = 1;
constexpr int32_t kFlagInclusive = 2;

size_t dispatch_clear_bytes(int64_t P) {
  return sizeof(WsHeader) + align_up(static_cast<size_t>(dispatch_blocks(P)) * sizeof(int32_t));
}

size_t dispatch_state_bytes(int64_t P, int E) {
  const size_t nb = static_cast<size_t>(dispatch_blocks(P));
  return align_up(nb * sizeof(int32_t)) + 2 * align_up(nb * static_cast<size_t>(E) * sizeof(int32_t));
}

DispatchState dispatch_state_at(void* base, int64_t P, int E) {
  const size_t nb = static_cast<size_t>(dispatch_blocks(P));
  char* p = static_cast<char*>(base);
  DispatchState st;
  st.flags = reinterpret_cast<int32_t*>(p);
  p += align_up(nb * sizeof(int32_t));
  st.agg = reinterpret_cast<int32_t*>(p);
  p += align_up(nb * static_cast<size_t>(E) * sizeof(int32_t));
  st.incl = reinterpret_cast<int32_t*>(p);
  return st;
}

namespace {

__device__ __forceinline__ int32_t load_acquire(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void store_release(int32_t* p, int32_t v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__global__ void __launch_bounds__(256) histogram_kernel(const int32_t* __restrict__ idx, int64_t P, int E,
                                                        int32_t* __restrict__ counts, int32_t* status) {
  extern __shared__ int32_t s_hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
  __syncthreads();
  bool bad = false;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p < P; p += stride) {
    const int e = __ldg(idx + p);
    if (e >= 0 && e < E)
      atomicAdd(&s_hist[e], 1);
    else
      bad = true;
  }
  if (bad) record_status(status, kStatusBadIndex);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = s_hist[e];
    if (c) atomicAdd(&counts[e], c);
  }
}

// Exclusive scan of s_in[0..n) into s_out[0..n], s_out[n] = total, by one
// block of kDispatchThreads threads.
__device__ void block_exclusive_scan(const int32_t* s_in, int32_t* s_out, int n, int32_t* s_tmp) {
  const int tid = threadIdx.x;
  const int per = (n + kDispatchThreads - 1) / kDispatchThreads;
  const int lo = tid * per;
  const int hi = min(n, lo + per);
  int32_t sum = 0;
  for (int i = lo; i < hi; ++i) sum += s_in[i];
  // inclusive scan of the per-thread sums
  const int lane = tid & 31, warp = tid >> 5;
  int32_t v = sum;
#pragma unroll
  for (int s = 1; s < 32; s <<= 1) {
    const int32_t o = __shfl_up_sync(0xffffffffu, v, s);
    if (lane >= s) v += o;
  }
  if (lane == 31) s_tmp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int32_t w = (lane < kWarps) ? s_tmp[lane] : 0;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, w, s);
      if (lane >= s) w += o;
    }
    if (lane < kWarps) s_tmp[lane] = w;
  }
  __syncthreads();
  int32_t run = v - sum + (warp > 0 ? s_tmp[warp - 1] : 0);
  for (int i = lo; i < hi; ++i) {
    s_out[i] = run;
    run += s_in[i];
  }
  if (tid == kDispatchThreads - 1) s_out[n] = s_tmp[kWarps - 1];
  __syncthreads();
}

__global__ void __launch_bounds__(kDispatchThreads)
index_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int64_t P, int E, int k,
             const int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ src_token,
             int32_t* __restrict__ dest_row, float* __restrict__ row_w, WsHeader* hdr, int32_t* flags,
             int32_t* agg, int32_t* incl) {
  extern __shared__ int32_t smem[];
  int32_t* s_cnt = smem;                    // [E]
  int32_t* s_off = s_cnt + E;               // [E+1]
  int32_t* s_warp = s_off + E + 1;          // [kWarps][E]: per-warp counts, then per-warp bases
  int32_t* s_agg = s_warp + kWarps * E;     // [E]: this block's per-expert totals
  int32_t* s_excl = s_agg + E;              // [E]: pairs of earlier blocks per expert
  __shared__ int32_t s_tmp[kWarps];
  __shared__ int32_t s_block;
  __shared__ int32_t s_flag;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_block = atomicAdd(&hdr->ticket, 1);
  for (int e = tid; e < E; e += kDispatchThreads) {
    s_cnt[e] = __ldcg(counts + e);
    s_excl[e] = 0;
  }
  for (int i = tid; i < kWarps * E; i += kDispatchThreads) s_warp[i] = 0;
  __syncthreads();
  const int64_t b = s_block;
  // this thread's pairs and gates, all in flight before the scan below
  const int64_t base = b * kDispatchChunk + static_cast<int64_t>(warp) * (32 * kDispatchPairsPerThread);
  int my_e[kDispatchPairsPerThread];
  float my_w[kDispatchPairsPerThread];
#pragma unroll
  for (int r = 0; r < kDispatchPairsPerThread; ++r) {
    const int64_t p = base + r * 32 + lane;
    my_e[r] = (p < P) ? __ldcg(topk_idx + p) : -1;
    my_w[r] = (p < P && row_w) ? __ldcg(topk_w + p) : 0.0f;
  }
  block_exclusive_scan(s_cnt, s_off, E, s_tmp);
  if (b == 0)
    for (int e = tid; e <= E; e += kDispatchThreads) offsets[e] = s_off[e];

  // rank each pair among the earlier pairs of its warp with the same expert
  int my_rank[kDispatchPairsPerThread];
  bool bad = false;
  const unsigned lanes_below = (1u << lane) - 1u;
#pragma unroll
  for (int r = 0; r < kDispatchPairsPerThread; ++r) {
    const int64_t p = base + r * 32 + lane;
    int e = my_e[r];
    if (p < P && (e < 0 || e >= E)) {
      bad = true;
      e = -1;
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    int rank = 0;
    if (e >= 0) rank = s_warp[warp * E + e] + __popc(same & lanes_below);
    __syncwarp();
    if (e >= 0 && lane == __ffs(same) - 1) s_warp[warp * E + e] += __popc(same);
    __syncwarp();
    my_e[r] = e;
    my_rank[r] = rank;
  }
  if (bad) record_status(&hdr->status, kStatusBadIndex);
  __syncthreads();

  // per-warp bases inside the block and the block's aggregate
  for (int e = tid; e < E; e += kDispatchThreads) {
    int32_t run = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int32_t c = s_warp[w * E + e];
      s_warp[w * E + e] = run;
      run += c;
    }
    s_agg[e] = run;
    (b == 0 ? incl : agg)[b * E + e] = run;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) store_release(&flags[b], b == 0 ? kFlagInclusive : kFlagAggregate);

  // decoupled look-back over the earlier blocks, a window of 32 at a time:
  // warp 0 reads the flags of blocks hi, hi-1, ..., hi-31 at once and waits
  // (bounded) until each has published at least its aggregate; the block
  // then adds the vectors of the blocks from hi down to the nearest one that
  // has published its inclusive prefix, or of the whole window, and goes on
  // below it.  Block 0 publishes its inclusive prefix first, so the walk
  // ends there at the latest.
  if (b > 0) {
    int64_t hi = b - 1;
    for (;;) {
      if (warp == 0) {
        const int64_t c = hi - lane;
        int32_t f = (c >= 0) ? load_acquire(flags + c) : kFlagAggregate;
        if (__any_sync(0xffffffffu, f == 0)) {
          const uint64_t t0 = global_timer_ns();
          for (;;) {
            __nanosleep(64);
            if (f == 0) f = load_acquire(flags + c);
            if (!__any_sync(0xffffffffu, f == 0)) break;
            if (__any_sync(0xffffffffu, global_timer_ns() - t0 > kWaitLimitNs)) {
              if (f == 0) f = -1;
              break;
            }
          }
        }
        const unsigned inclusive = __ballot_sync(0xffffffffu, c >= 0 && f == kFlagInclusive);
        const bool lost = __any_sync(0xffffffffu, f < 0);
        // lane of the nearest inclusive block, 32 when the window has none
        if (lane == 0) s_flag = lost ? -1 : (inclusive ? __ffs(inclusive) - 1 : 32);
      }
      __syncthreads();
      const int32_t stop = s_flag;
      if (stop < 0) {
        if (tid == 0) record_status(&hdr->status, kStatusTimeout);
        // this block's pairs get no row: -1 tells the permute and the
        // combine to skip them (their rows in the expert groups stay unwritten)
#pragma unroll
        for (int r = 0; r < kDispatchPairsPerThread; ++r) {
          const int64_t p = base + r * 32 + lane;
          if (p < P) dest_row[p] = -1;
        }
        return;  // successors walk past this block on its aggregate
      }
      // every load of the window in flight at once: one L2 round trip
      const int n_agg = min(stop, 32);
      for (int e = tid; e < E; e += kDispatchThreads) {
        int32_t part[33];
#pragma unroll
        for (int i = 0; i < 32; ++i) part[i] = (i < n_agg) ? __ldcg(agg + (hi - i) * E + e) : 0;
        part[32] = (stop < 32) ? __ldcg(incl + (hi - stop) * E + e) : 0;
        int32_t acc = 0;
#pragma unroll
        for (int i = 0; i < 33; ++i) acc += part[i];
        s_excl[e] += acc;
      }
      __syncthreads();  // s_flag is rewritten next round
      if (stop < 32) break;
      hi -= 32;
    }
    for (int e = tid; e < E; e += kDispatchThreads) incl[b * E + e] = s_excl[e] + s_agg[e];
    __threadfence();
    __syncthreads();
    if (tid == 0) store_release(&flags[b], kFlagInclusive);
  }

  // rows: expert base + earlier blocks + earlier warps + rank within the warp
#pragma unroll
  for (int r = 0; r < kDispatchPairsPerThread; ++r) {
    const int64_t p = base + r * 32 + lane;
    if (p >= P) continue;
    const int e = my_e[r];
    if (e < 0) {
      dest_row[p] = -1;
      continue;
    }
    const int32_t row = s_off[e] + s_excl[e] + s_warp[warp * E + e] + my_rank[r];
    dest_row[p] = row;
    src_token[row] = static_cast<int32_t>(p / k);
    if (row_w) row_w[row] = my_w[r];
  }
}

}  // namespace

cudaError_t launch_histogram(const int32_t* topk_idx, int64_t P, int E, int32_t* counts, int32_t* status,
                             int num_sms, cudaStream_t stream) {
  if (P == 0) return cudaSuccess;
  const int64_t want = (P + 255) / 256;
  const int grid = static_cast<int>(want < num_sms * 4 ? want : num_sms * 4);
  histogram_kernel<<<grid, 256, E * sizeof(int32_t), stream>>>(topk_idx, P, E, counts, status);
  return cudaGetLastError();
}

cudaError_t launch_index(const int32_t* topk_idx, const float* topk_w, int64_t P, int E, int k,
                         const int32_t* counts, int32_t* offsets, int32_t* src_token, int32_t* dest_row,
                         float* row_w, void* header, DispatchState st, cudaStream_t stream) {
  const int64_t nb = dispatch_blocks(P);
  if (nb == 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(E + (E + 1) + kWarps * E + E + E) * sizeof(int32_t);
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(index_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
  }
  index_kernel<<<static_cast<unsigned>(nb), kDispatchThreads, smem, stream>>>(
      topk_idx, topk_w, P, E, k, counts, offsets, src_token, dest_row, row_w, static_cast<WsHeader*>(header),
      st.flags, st.agg, st.incl);
  return cudaGetLastError();
}

}  // namespace moe
