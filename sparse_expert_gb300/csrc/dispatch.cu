// Stages 2 and 3 of the layer: per-expert token counts, their prefix sums,
// and the index maps ("Scalable Pretraining of Large MoE LMs on Aurora
// Super Computer", §3.1, Algorithm 1, stages 2-3).
//
// The page's kernels give each thread a block of tokens, count per
// (expert, thread), prefix-sum the expert-major count table, and let each
// (expert, thread) write rows from its base with a running counter.  The
// result is a stable counting sort of the pairs by expert.  Here the same
// sort is done by chunks of 2,048 consecutive pairs:
//   1. a table of per-chunk counts, hist[c][e]: the route kernel adds each
//      pair it selects into it (the forward), or a histogram kernel writes
//      one chunk's row per block (moe_dispatch_scan);
//   2. one pass, one block per chunk: the block sums the table's columns --
//      over every chunk for the expert totals (the counts, and the offsets
//      by an exclusive scan), over the chunks before its own for its
//      per-expert base -- ranks its pairs within the chunk (warp match +
//      per-warp running counts) and writes every pair's row.
// The table is complete before the pass starts, so no block ever waits for
// another: the pass is one round of loads, a scan and the writes.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kWarps = kDispatchThreads / 32;

int dispatch_hist_stride(int E) { return (E + 3) & ~3; }

size_t dispatch_hist_bytes(int64_t P, int E) {
  return align_up(static_cast<size_t>(dispatch_blocks(P)) * dispatch_hist_stride(E) * sizeof(int32_t));
}

namespace {

// One chunk's row of the count table, written in full (zeros included), so
// the table needs no clearing.
__global__ void __launch_bounds__(kDispatchThreads)
chunk_histogram_kernel(const int32_t* __restrict__ idx, int64_t P, int E, int E4, int32_t* __restrict__ hist,
                       int32_t* status) {
  extern __shared__ int32_t s_hist[];
  for (int e = threadIdx.x; e < E4; e += kDispatchThreads) s_hist[e] = 0;
  __syncthreads();
  bool bad = false;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kDispatchChunk;
#pragma unroll
  for (int r = 0; r < kDispatchPairsPerThread; ++r) {
    const int64_t p = base + r * kDispatchThreads + threadIdx.x;
    if (p < P) {
      const int e = __ldg(idx + p);
      if (e >= 0 && e < E)
        atomicAdd(&s_hist[e], 1);
      else
        bad = true;
    }
  }
  if (bad) record_status(status, kStatusBadIndex);
  __syncthreads();
  int32_t* row = hist + static_cast<int64_t>(blockIdx.x) * E4;
  for (int e = threadIdx.x; e < E4; e += kDispatchThreads) row[e] = s_hist[e];
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

__device__ __forceinline__ int4 add4(int4 a, int4 b) { return make_int4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }

__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

__global__ void __launch_bounds__(kDispatchThreads)
index_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int64_t P, int E, int E4, int k,
             const int32_t* __restrict__ hist, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
             int32_t* __restrict__ src_token, int32_t* __restrict__ dest_row, float* __restrict__ row_w,
             int32_t* status, int slab_rows) {
  extern __shared__ __align__(16) int32_t smem[];
  int4* s_slab = reinterpret_cast<int4*>(smem);      // [slab_rows][E4 / 4]: rows of the count table
  int32_t* s_tot = smem + slab_rows * E4;   // [E4]: pairs per expert
  int32_t* s_excl = s_tot + E4;             // [E4]: pairs of earlier chunks per expert
  int32_t* s_off = s_excl + E4;             // [E+1]
  int32_t* s_warp = s_off + E + 1;          // [kWarps][E]: per-warp counts, then per-warp bases
  __shared__ int4 s_part[2][kDispatchThreads];  // column partial sums of each row group: totals, earlier chunks
  __shared__ int32_t s_tmp[kWarps];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int nchunks = gridDim.x;
  // this thread's pairs and gates, in flight before the column sums below
  const int64_t base = static_cast<int64_t>(b) * kDispatchChunk + static_cast<int64_t>(warp) * (32 * kDispatchPairsPerThread);
  int my_e[kDispatchPairsPerThread];
  float my_w[kDispatchPairsPerThread];
#pragma unroll
  for (int r = 0; r < kDispatchPairsPerThread; ++r) {
    const int64_t p = base + r * 32 + lane;
    my_e[r] = (p < P) ? __ldcg(topk_idx + p) : -1;
    my_w[r] = (p < P && row_w) ? __ldcg(topk_w + p) : 0.0f;
  }
  for (int i = tid; i < kWarps * E; i += kDispatchThreads) s_warp[i] = 0;

  // column sums of the count table, four experts per 16-byte word: the
  // table comes into shared memory in slabs of slab_rows rows, every copy of
  // a slab in flight at once (cp.async), and thread (row group g, column
  // quad q) adds rows g, g + G, ... of the slab; the G row groups are then
  // added in shared memory
  const int Q = E4 / 4;
  const int G = kDispatchThreads / Q;  // >= 1: E4 <= 1024
  const int q = tid % Q, g = tid / Q;
  const int4* h4 = reinterpret_cast<const int4*>(hist);
  int4 tot = make_int4(0, 0, 0, 0), ex = make_int4(0, 0, 0, 0);
  for (int r0 = 0; r0 < nchunks; r0 += slab_rows) {
    const int rows = min(slab_rows, nchunks - r0);
    const int words = rows * Q;
    for (int i = tid; i < words; i += kDispatchThreads) cp_async_16(s_slab + i, h4 + static_cast<int64_t>(r0) * Q + i);
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    if (g < G) {
      for (int r = g; r < rows; r += G) {
        const int4 v = s_slab[r * Q + q];
        tot = add4(tot, v);
        if (r0 + r < b) ex = add4(ex, v);
      }
    }
    __syncthreads();
  }
  if (g < G) {
    s_part[0][tid] = tot;
    s_part[1][tid] = ex;
  }
  __syncthreads();
  for (int qq = tid; qq < Q; qq += kDispatchThreads) {
    int4 col_tot = s_part[0][qq], col_ex = s_part[1][qq];
    for (int gg = 1; gg < G; ++gg) {
      col_tot = add4(col_tot, s_part[0][gg * Q + qq]);
      col_ex = add4(col_ex, s_part[1][gg * Q + qq]);
    }
    reinterpret_cast<int4*>(s_tot)[qq] = col_tot;
    reinterpret_cast<int4*>(s_excl)[qq] = col_ex;
  }
  __syncthreads();
  if (b == 0)
    for (int e = tid; e < E; e += kDispatchThreads) counts[e] = s_tot[e];
  block_exclusive_scan(s_tot, s_off, E, s_tmp);
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
  if (bad) record_status(status, kStatusBadIndex);
  __syncthreads();

  // per-warp bases inside the chunk
  for (int e = tid; e < E; e += kDispatchThreads) {
    int32_t run = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int32_t c = s_warp[w * E + e];
      s_warp[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();

  // rows: expert base + earlier chunks + earlier warps + rank within the warp
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

cudaError_t launch_chunk_histogram(const int32_t* topk_idx, int64_t P, int E, int32_t* hist, int32_t* status,
                                   cudaStream_t stream) {
  const int64_t nb = dispatch_blocks(P);
  if (nb == 0) return cudaSuccess;
  const int E4 = dispatch_hist_stride(E);
  chunk_histogram_kernel<<<static_cast<unsigned>(nb), kDispatchThreads, E4 * sizeof(int32_t), stream>>>(
      topk_idx, P, E, E4, hist, status);
  return cudaGetLastError();
}

cudaError_t launch_index(const int32_t* topk_idx, const float* topk_w, int64_t P, int E, int k, const int32_t* hist,
                         int32_t* counts, int32_t* offsets, int32_t* src_token, int32_t* dest_row, float* row_w,
                         int32_t* status, cudaStream_t stream) {
  const int64_t nb = dispatch_blocks(P);
  if (nb == 0) return cudaSuccess;
  const int E4 = dispatch_hist_stride(E);
  // slabs of the count table up to 96 KB (the whole table up to 2^17 pairs at
  // E = 384), beside the block's other shared arrays
  const int64_t row_bytes = static_cast<int64_t>(E4) * sizeof(int32_t);
  const int slab_rows = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(nb, (96 * 1024) / row_bytes)));
  const size_t smem = static_cast<size_t>(slab_rows) * row_bytes +
                      static_cast<size_t>(E4 + E4 + (E + 1) + kWarps * E) * sizeof(int32_t);
  // the static arrays (column partial sums, scan scratch) count against the same 48 KB default
  constexpr size_t kStaticSmem = 2 * kDispatchThreads * sizeof(int4) + kWarps * sizeof(int32_t);
  if (smem + kStaticSmem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(index_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
  }
  index_kernel<<<static_cast<unsigned>(nb), kDispatchThreads, smem, stream>>>(
      topk_idx, topk_w, P, E, E4, k, hist, counts, offsets, src_token, dest_row, row_w, status, slab_rows);
  return cudaGetLastError();
}

}  // namespace moe
