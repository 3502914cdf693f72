// Grouped expert GEMMs on SM pairs (tcgen05 cta_group::2, sm_103a), with
// the weights as the 256-row operand and the tokens as N: the forward's two
// GEMMs and the backward's two dgrad GEMMs.
//
// "Scalable Pretraining of Large MoE LMs on Aurora Super Computer", §3.1,
// Algorithm 1, stage 4: gate_out/up_out = Grouped_mm(mlp_in, weight);
// mul_out = Silu(gate_out) * up_out; mlp_out = Grouped_mm(mul_out,
// down_weight), over expert-contiguous rows bounded by the cumulative
// token counts; and the same stage differentiated for the activations:
// dH = dY Wd^T with dG = dH U Silu'(G), dU = dH Silu(G); dX = [dG | dU]
// [Wg ; Wu]^T.
//
// Each tile computes D^T = W_e[256 rows, K] x X_e[N tokens, K]^T on a pair
// of SMs (a 2-CTA cluster) for up to 512 of the expert's tokens at once
// (all of them at the 1T layer's ~341 per expert), so every weight tile is
// read once per expert.  Per K step the leader issues tcgen05.mma M=256 with
// N1 = min(N, 256) tokens and, when N > 256, a second one with the other
// N2 = N - 256 into the next TMEM columns; N is the tile's token count
// rounded up to 16.  CTA r holds 128 weight rows and, of each part, the
// token rows r*N_part/2 .. +N_part/2 (128-row boxes).  The accumulator lands
// in each CTA's TMEM as its 128 weight rows x N token columns.  Per SM this
// takes in 8.3 KB of operands per MFLOP (a one-SM 128 x 256 tile: 11.4).
// One accumulator: the epilogue drains a tile before the next one starts.
// The forward reads the packed weights K-major; the dgrad GEMMs read the
// same packed tiles transposed (MN-major A: two consecutive 64-column
// blocks of a packed tile per CTA and K block).
//
// Epilogues (each warp: 32 TMEM lanes = weight rows, 32-token chunks,
// loaded as two 16x256b blocks whose fragment is stmatrix's, staged as
// token rows in shared memory so every global access covers whole
// token-row segments):
//   gate/up: a tile's 256 weight rows are two packed gate/up tiles of 64
//     gate then the same 64 up columns, one per CTA, loaded by a 4-D tensor
//     map in quarter order: each 32-lane TMEM quadrant holds 16 gate
//     features and, 16 lanes further on, the same 16 up features, so each
//     warp forms Silu(gate)*up in fp32 from its own two 16-lane loads and
//     stores H[token, j] for its 16 features (and, for the backward's
//     recomputation, the raw G and U in the packed column order);
//   rows: Y[token, i] or dX[token, i] as they are, or scaled by a gate per
//     token; a warp reads its last kHold chunks into registers (bf16) before
//     it hands the accumulator back, so their stores overlap the next
//     tile's MMAs;
//   SwiGLU backward: dH with the saved G, U of the same rows (ldmatrix.trans
//     turns their token rows into the fragment), stores dG and dU.
//
// The kernel is instantiated once per epilogue, so that each gets the
// registers of its own epilogue (10 warps: at most 168 per thread).
//
// Roles in each CTA of the pair (320 threads): warp 0 TMA producer (both
// CTAs load their halves; every copy signals the leader's stage barrier),
// warp 1 MMA issuer (leader only; its commits are multicast to both CTAs),
// warps 2-9 epilogue, two per TMEM lane quadrant, each draining half of the
// tile's token chunks.  Tiles come from a shared atomic counter (dynamic
// scheduling): the leader claims each tile and writes its id into both
// CTAs' rings, over a flat order expert -> weight tile -> token tile
// (consecutive tiles share a weight tile in L2; an expert's tokens stay in
// L2 across its weight tiles).  Every wait is bounded; a CTA that gives up
// records a timeout, and both CTAs meet at a cluster barrier before TMEM is
// released.
#include <cuda.h>

#include "common.cuh"
#include "gemm_common.cuh"
#include "pair_common.cuh"
#include "internal.h"
#include "moe_gb300.h"

namespace moe {

// the paired GEMMs' tile schedule for this process (set through the C ABI
// for measurement; dynamic by default)
static bool g_static_tiles = false;

namespace {

constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int kTileN = 512;       // tokens per tile (both CTAs): up to two MMAs of N <= 256
constexpr int kPartN = 256;       // N of one MMA
constexpr int kHalfRows = 128;    // weight rows and token rows (per part) staged per CTA
constexpr int kABytes = kHalfRows * BK * 2;
constexpr int kBBytes = kHalfRows * BK * 2;          // one token part
constexpr int kStageBytes = kABytes + 2 * kBBytes;   // A | B part 1 | B part 2
constexpr int kEpiParts = 2;     // epilogue warps per TMEM lane quadrant, each a share of the token chunks
constexpr int kEpiWarps = 4 * kEpiParts;
constexpr int kTmemCols = 512;    // one accumulator: the tile's weight rows x up to 512 tokens
constexpr int kEpiBytes = kEpiWarps * 32 * 64;   // per epilogue warp 2 KB: the staging of its stores
constexpr int kRing = 4;                          // tile ids published ahead
constexpr int kCodeBytes = kHalfRows * BK;        // FP8 codes of one CTA's weight rows and K block

// Per-instantiation layout.  The bf16 form has one ring of stages, each
// A | B part 1 | B part 2.  The FP8-weight form adds four converter warps
// (a slice of a weight row per thread) and a code-producer warp, and splits
// the ring: a ring of A slots that the converters fill (four deep, so a
// slot is converted, fenced and signalled across the pair while the MMA
// works through the three before it), a ring of token stages (B parts 1 and
// 2, three deep) and a ring of code stages (8 KB of 64-byte-swizzled codes
// and one scale record each), all within 227 KB of shared memory.
template <bool kFp8>
struct Cfg {
  static constexpr int kStages = kFp8 ? 3 : 4;                         // stages of the producer's ring
  static constexpr int kSlotBytes = kFp8 ? 2 * kBBytes : kStageBytes;  // one stage of that ring
  static constexpr int kAStages = kFp8 ? 4 : 0;                        // A slots the converters fill
  // A slots per cluster-scope release of the peer's signaller: the release
  // is the one serial step per stage that crosses the pair, so it covers two
  // slots (K blocks come in pairs: the FP8 form needs K % 128 == 0)
  static constexpr int kSigGroup = 2;
  static constexpr int kConvWarps = kFp8 ? 4 : 0;
  static constexpr int kCodeWarps = kFp8 ? 1 : 0;
  static constexpr int kCodeStages = kFp8 ? 4 : 0;
  static constexpr int kCodeStageBytes = 9216;  // codes + a scale record, rounded to 1 KB
  static constexpr int kThreads = 64 + 32 * (kEpiWarps + kConvWarps + kCodeWarps);
  // readers of a ring slot, counted on the leader's rempty: the leader's MMA
  // thread, the peer's producer, both CTAs' epilogue, converter and
  // code-producer warps, and with FP8 weights the peer's signaller
  static constexpr int kRingReaders = 2 + 2 * (kEpiWarps + kConvWarps + kCodeWarps) + (kFp8 ? 1 : 0);
  // chunks an epilogue warp holds in registers across the hand-back, row
  // epilogue and gate/up epilogue (the FP8 form has more warps, so fewer
  // registers per thread)
  static constexpr int kHold = kFp8 ? (kConvWarps > 4 ? 2 : 4) : 6;
  static constexpr int kHoldH = kFp8 && kConvWarps > 4 ? 2 : 4;
};

// What the epilogue makes of the accumulator (weight rows x token columns)
enum : int {
  kModeSwiGLU = 0,     // gate/up: H = Silu(G) * U (and optionally G, U themselves)
  kModeRows = 1,       // the rows as they are (down, dX), optionally scaled per token
  kModeSwiGLUBwd = 2,  // dH: dG = dH U Silu'(G), dU = dH Silu(G) from the saved G, U
};

struct Params {
  const int32_t* offsets;
  const float* row_scale;  // kModeRows, kModeSwiGLUBwd: gate of each row, or null
  __nv_bfloat16* out;      // H [P, f], Y [P, d], dX [P, d] or dG,dU [P, 2f] (packed interleave)
  __nv_bfloat16* gu;       // kModeSwiGLU: also G, U [P, 2f] in the packed interleave, or null
  const __nv_bfloat16* gu_in;  // kModeSwiGLUBwd: the saved G, U [P, 2f]
  __nv_bfloat16* dh_out;       // kModeSwiGLUBwd: also the accumulator as it is (dH before row_scale) [P, f], or null
  int32_t* status;
  int32_t* tile_counter;   // zeroed before launch
  int E;
  int K;
  int m_tiles;         // 256-row weight tiles per expert
  int a_tile_rows;     // rows of one packed weight tile (128 gate/up, 256 down)
  int a_tiles;         // packed weight tiles per expert
  int a_mn;            // weights read transposed: M runs along a packed tile's columns
  int a_mblocks;       // a_mn: 64-column blocks of one packed tile
  int out_cols;        // f or d (kModeSwiGLUBwd: f, rows of 2f)
  int mode;
  // FP8 weights: the codes come through the weight tensor map (64-byte rows
  // of 128-row tiles), the scale records from here
  const float* scales;  // records of rec_floats floats, one per (expert, scale tile, K block)
  int code_tiles;       // 128-row code tiles per expert
  int sc_tiles;         // scale tiles per expert
  int sc_per_cta;       // 1: each CTA of a pair has its own scale tile (down); 0: one per pair (gate/up)
  int rec_floats;
  int static_tiles;     // 1: pair i takes tiles i, i + pairs, ... (measurement); 0: a shared counter
};

template <bool kFp8>
struct SmemT {
  uint64_t full[Cfg<kFp8>::kStages], empty[Cfg<kFp8>::kStages];
  uint64_t cfull[kFp8 ? Cfg<kFp8>::kCodeStages : 1], cempty[kFp8 ? Cfg<kFp8>::kCodeStages : 1];
  uint64_t converted[kFp8 ? Cfg<kFp8>::kAStages : 1];  // this CTA's converter warps have written an A slot
  uint64_t apeer[kFp8 ? Cfg<kFp8>::kAStages : 1];      // leader: the peer's A slot is written (its signaller)
  uint64_t aempty[kFp8 ? Cfg<kFp8>::kAStages : 1];     // the MMA is done with an A slot
  uint64_t tfull[2], tempty[2];
  uint64_t rfull[kRing], rempty[kRing];
  int32_t ring[kRing];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Tile t: expert, weight tile, token tile.  s_pre[e] = tiles of experts
// before e; an expert has m_tiles x ceil(rows / 512) tiles, token tile
// fastest.
struct Tile {
  int e, mt, nt, tok0, valid, n;
};

// An expert's rows are split into ceil(rows / 512) near-equal token tiles
// of S rows (a multiple of 16, at most 512); returns the tile count and
// sets S.
__host__ __device__ __forceinline__ int token_tiles(int rows, int& S) {
  if (rows <= 0) {
    S = 0;
    return 0;
  }
  const int n0 = (rows + kTileN - 1) / kTileN;
  S = (((rows + n0 - 1) / n0) + 15) & ~15;
  return (rows + S - 1) / S;  // every tile holds at least one row
}

__device__ __forceinline__ Tile decode(int t, const int32_t* s_off, const int32_t* s_pre, int E, int m_tiles) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pre[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  Tile x;
  x.e = lo;
  const int rows = s_off[lo + 1] - s_off[lo];
  int S;
  const int ntt = token_tiles(rows, S);
  const int local = t - s_pre[lo];
  x.mt = local / ntt;
  x.nt = local - x.mt * ntt;
  x.tok0 = s_off[lo] + x.nt * S;
  x.valid = min(S, rows - x.nt * S);
  x.n = (x.valid + 15) & ~15;
  (void)m_tiles;
  return x;
}

// A warp's token-row staging buffer: up to 32 token rows of 64 bytes (the
// warp's 32 bf16 features), the 16-byte pieces of row t swizzled by
// (t >> 1) & 3 so that the stmatrix writes and the 16-byte row reads are
// both free of bank conflicts.
//
// p[4g + m] holds features 8m .. 8m+7 of tokens 8g .. 8g+7 as an stmatrix
// fragment: thread i has feature 8m + i/4 of tokens 8g + 2(i%4) and +1,
// packed low/high -- which is what packing the columns of a 16x256b TMEM
// load (features = TMEM lanes, tokens = TMEM columns) pairwise gives.
template <int G>
__device__ __forceinline__ void stage_rows(const uint32_t (&p)[4 * G], uint8_t* buf, int lane) {
  const uint32_t a0 = smem_addr(buf) + (lane & 7) * 64 + ((((lane >> 3) ^ (lane >> 1)) & 3) << 4);
#pragma unroll
  for (int g = 0; g < G; ++g) stmatrix_x4_trans(a0 + g * 512, p[4 * g], p[4 * g + 1], p[4 * g + 2], p[4 * g + 3]);
  __syncwarp();
}

// Rows 0 .. ROWS-1 of the staging buffer to out rows 0 .. ROWS-1 (row
// stride ld), rows >= valid skipped: each 16-byte store instruction covers
// 8 rows x 64 contiguous bytes.
template <int ROWS>
__device__ __forceinline__ void rows_to_global(const uint8_t* buf, int lane, __nv_bfloat16* out, int64_t ld,
                                               int valid) {
  constexpr int kPer = ROWS * 4 / 32;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int idx = i * 32 + lane;
    const int r = idx >> 2;
    const int q = idx & 3;
    const uint4 v = *reinterpret_cast<const uint4*>(buf + r * 64 + ((q ^ ((r >> 1) & 3)) << 4));
    if (r < valid) *reinterpret_cast<uint4*>(out + r * ld + q * 8) = v;
  }
  __syncwarp();
}

// rows_to_global with the row's first 32 bytes going to out and its last
// 32 bytes to out + hi (elements).
__device__ __forceinline__ void rows_to_global_split(const uint8_t* buf, int lane, __nv_bfloat16* out, int hi,
                                                     int64_t ld, int valid) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int idx = i * 32 + lane;
    const int r = idx >> 2;
    const int q = idx & 3;
    const uint4 v = *reinterpret_cast<const uint4*>(buf + r * 64 + ((q ^ ((r >> 1) & 3)) << 4));
    if (r < valid) *reinterpret_cast<uint4*>(out + r * ld + (q < 2 ? q * 8 : hi + (q - 2) * 8)) = v;
  }
  __syncwarp();
}

// A warp's 16-feature staging buffer: 32 token rows of 32 bytes, the
// 16-byte half h of row t at position h ^ ((t >> 2) & 1), so that both the
// stmatrix writes and the row reads are free of bank conflicts.  p[2g + m]
// holds features 8m .. 8m+7 of tokens 8g .. 8g+7 as an stmatrix fragment
// (thread i: feature 8m + i/4 of tokens 8g + 2(i%4) and +1).
__device__ __forceinline__ void stage_rows_16f(const uint32_t (&p)[8], uint8_t* buf, int lane) {
  const int j = lane >> 3;  // the matrix of each x4 whose row this lane addresses: (m = j & 1, g = 2s + j / 2)
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int r = 8 * (2 * s + (j >> 1)) + (lane & 7);
    stmatrix_x4_trans(smem_addr(buf) + r * 32 + (((j & 1) ^ ((r >> 2) & 1)) << 4), p[4 * s], p[4 * s + 1],
                      p[4 * s + 2], p[4 * s + 3]);
  }
  __syncwarp();
}

// Rows 0 .. 31 of a 16-feature staging buffer to out (row stride ld), rows
// >= valid skipped: each 16-byte store instruction covers 16 rows x 32 bytes.
__device__ __forceinline__ void rows16f_to_global(const uint8_t* buf, int lane, __nv_bfloat16* out, int64_t ld,
                                                  int valid) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int idx = i * 32 + lane;
    const int r = idx >> 1;
    const int q = idx & 1;
    const uint4 v = *reinterpret_cast<const uint4*>(buf + r * 32 + ((q ^ ((r >> 2) & 1)) << 4));
    if (r < valid) *reinterpret_cast<uint4*>(out + r * ld + q * 8) = v;
  }
  __syncwarp();
}

// 16 token rows of a 64-byte column segment of src (row stride ld; rows
// >= valid as zeros) into two 16-byte registers per thread, and from there
// into the staging buffer (8 rows x 64 contiguous bytes per load
// instruction): split so the loads can be issued early.
__device__ __forceinline__ void load_rows16(uint4 (&v)[2], int lane, const __nv_bfloat16* src, int64_t ld,
                                            int valid) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int idx = i * 32 + lane;
    const int r = idx >> 2;
    const int q = idx & 3;
    v[i] = r < valid ? __ldg(reinterpret_cast<const uint4*>(src + r * ld + q * 8)) : make_uint4(0, 0, 0, 0);
  }
}
__device__ __forceinline__ void store_rows16(uint8_t* buf, int lane, const uint4 (&v)[2]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int idx = i * 32 + lane;
    const int r = idx >> 2;
    const int q = idx & 3;
    *reinterpret_cast<uint4*>(buf + r * 64 + ((q ^ ((r >> 1) & 3)) << 4)) = v[i];
  }
  __syncwarp();
}

// The inverse of stage_rows: ldmatrix .trans hands thread i features
// 8m + i/4 of tokens 8g + 2(i%4) and +1 (p[4g + m], packed low/high).
template <int G>
__device__ __forceinline__ void rows_to_fragment(const uint8_t* buf, int lane, uint32_t (&p)[4 * G]) {
  const uint32_t a0 = smem_addr(buf) + (lane & 7) * 64 + ((((lane >> 3) ^ (lane >> 1)) & 3) << 4);
#pragma unroll
  for (int g = 0; g < G; ++g)
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(p[4 * g]), "=r"(p[4 * g + 1]), "=r"(p[4 * g + 2]), "=r"(p[4 * g + 3])
                 : "r"(a0 + g * 512)
                 : "memory");
  __syncwarp();
}

// The fragment of a 32-feature x 32-token chunk from its two 16x256b loads
// (a: features 0-15, b: 16-31), rounded to bf16.
__device__ __forceinline__ void pack_chunk(const uint32_t (&a)[16], const uint32_t (&b)[16], uint32_t (&p)[16]) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    p[4 * g] = pack_bf16x2(__uint_as_float(a[4 * g]), __uint_as_float(a[4 * g + 1]));
    p[4 * g + 1] = pack_bf16x2(__uint_as_float(a[4 * g + 2]), __uint_as_float(a[4 * g + 3]));
    p[4 * g + 2] = pack_bf16x2(__uint_as_float(b[4 * g]), __uint_as_float(b[4 * g + 1]));
    p[4 * g + 3] = pack_bf16x2(__uint_as_float(b[4 * g + 2]), __uint_as_float(b[4 * g + 3]));
  }
}

// FP8 weights: the four E4M3 codes of `word` (byte i = code i) as exact
// fp32 values.  The hardware conversion of a code pair to f16 is exact
// (every E4M3 value, subnormals included, is an f16 value; the encoder
// never writes the NaN codes), and so is the widening of f16 to fp32.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t word, float (&v)[4]) {
  uint32_t h01, h23;
  asm("{.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, hi;}"
      : "=r"(h01), "=r"(h23)
      : "r"(word));
  asm("{.reg .f16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.f32.f16 %0, a;\n\t"
      "cvt.f32.f16 %1, b;}"
      : "=f"(v[0]), "=f"(v[1])
      : "r"(h01));
  asm("{.reg .f16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.f32.f16 %0, a;\n\t"
      "cvt.f32.f16 %1, b;}"
      : "=f"(v[2]), "=f"(v[3])
      : "r"(h23));
}

// Two fp32 products, each rounded once to nearest (one packed multiply),
// then both rounded to bf16.
__device__ __forceinline__ uint32_t mul_pair_to_bf16x2(float v0, float v1, float s0, float s1) {
  uint64_t vv, ss, pp;
  asm("mov.b64 %0, {%1, %2};" : "=l"(vv) : "f"(v0), "f"(v1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(ss) : "f"(s0), "f"(s1));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(pp) : "l"(vv), "l"(ss));
  float p0, p1;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(p0), "=f"(p1) : "l"(pp));
  return pack_bf16x2(p0, p1);
}

// One 16-value piece of a weight row of one K block: 16 E4M3 codes and
// their 16 scales become bf16(value x scale), the product of the exact code
// value and the fp32 scale rounded once in fp32 and then to bf16 -- the
// dequantisation of the "FP8 expert weight all-gather", bit for bit.
__device__ __forceinline__ void convert_piece(const uint4& q, const float4 (&scl)[4], uint32_t (&o)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float v[4];
    e4m3x4_to_f32(w[i], v);
    o[2 * i] = mul_pair_to_bf16x2(v[0], v[1], scl[i].x, scl[i].y);
    o[2 * i + 1] = mul_pair_to_bf16x2(v[2], v[3], scl[i].z, scl[i].w);
  }
}

// One instantiation per epilogue mode (and weight format), so that each gets
// the registers of its own epilogue.
template <int kMode, bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<kFp8>::kThreads, 1)
grouped_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                        const Params p) {
  using C = Cfg<kFp8>;
  using Smem = SmemT<kFp8>;
  constexpr int kStages = C::kStages;
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  uint8_t* s_stage0 = base;  // stage s at s_stage0 + s * kSlotBytes: [A |] B part 1 | B part 2
  uint8_t* s_a0 = s_stage0 + kStages * C::kSlotBytes;   // FP8: A slot a at s_a0 + a * kABytes
  uint8_t* s_code0 = s_a0 + C::kAStages * kABytes;      // FP8: code stage c at s_code0 + c * kCodeStageBytes
  uint8_t* s_epi = s_code0 + C::kCodeStages * C::kCodeStageBytes;
  Smem* S = reinterpret_cast<Smem*>(s_epi + kEpiBytes);
  int32_t* s_off = reinterpret_cast<int32_t*>(S + 1);
  int32_t* s_pre = s_off + (p.E + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
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
      int S;
      int v = p.m_tiles * token_tiles(hi - lo, S);
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
    tmem_alloc_pair(&S->tmem_base, kTmemCols);
  } else if (warp == 2 && lane == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&S->full[i], 1);  // the leader's producer: the bytes to come
      mbar_init(&S->empty[i], 1);
    }
    for (int i = 0; i < C::kCodeStages; ++i) {
      mbar_init(&S->cfull[i], 1);
      mbar_init(&S->cempty[i], C::kConvWarps);
    }
    for (int i = 0; i < C::kAStages; ++i) {
      mbar_init(&S->converted[i], C::kConvWarps);
      mbar_init(&S->apeer[i], 1);
      mbar_init(&S->aempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S->tfull[i], 1);
      mbar_init(&S->tempty[i], 2 * kEpiWarps);  // both CTAs' epilogue warps (leader's copy is used)
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&S->rfull[i], 1);
      mbar_init(&S->rempty[i], C::kRingReaders);  // the leader's copy is used
    }
    mbar_init(&S->drain, 1);
    S->abort = 0;
    fence_barrier_init();
  }
  tc_fence_before_sync();
  cluster_sync();
  tc_fence_after_sync();

  const int total = s_pre[p.E];
  const uint32_t tmem_base = S->tmem_base;
  bool failed = false;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      tma_prefetch_desc(&tm_x);
      const int num_kb = p.K / BK;
      int stage = 0;
      uint32_t phase = 0;
      int rs = 0;
      uint32_t rphase = 0;
      int claimed = 0;
      for (;;) {
        // tiles come from a shared counter (dynamic scheduling): the leader
        // claims one and publishes it in both CTAs' rings
        int t;
        if (rank == 0) {
          if (!wait_cluster(&S->rempty[rs], rphase ^ 1u, abort_flag)) {
            failed = true;
            break;
          }
          // static schedule (for measurement): pair i takes tiles i, i + pairs, ...
          t = p.static_tiles ? static_cast<int>(blockIdx.x >> 1) + claimed++ * static_cast<int>(gridDim.x >> 1)
                             : atomicAdd(p.tile_counter, 1);
          if (t >= total) t = -1;
          S->ring[rs] = t;
          st_cluster(pair_addr(&S->ring[rs], 1), t);
          mbar_arrive(&S->rfull[rs]);
          arrive_remote(pair_addr(&S->rfull[rs], 1));
        } else {
          if (!wait_cluster(&S->rfull[rs], rphase, abort_flag)) {
            failed = true;
            break;
          }
          t = S->ring[rs];
          arrive_remote(leader_addr(&S->rempty[rs]));
        }
        if (++rs == kRing) {
          rs = 0;
          rphase ^= 1u;
        }
        if (t < 0) break;
        const Tile x = decode(t, s_off, s_pre, p.E, p.m_tiles);
        // this CTA's 128 weight rows: packed tile and row inside it (K-major),
        // or, read transposed, the two 64-column blocks that hold them
        const int w0 = x.mt * 2 * kHalfRows + static_cast<int>(rank) * kHalfRows;
        const int wblk = (x.e * p.a_tiles + w0 / p.a_tile_rows) * num_kb;
        const int wrow = w0 % p.a_tile_rows;
        // this CTA's token rows of each part
        const int n1 = min(x.n, kPartN), n2 = x.n - n1;
        const int xrow1 = x.tok0 + static_cast<int>(rank) * (n1 >> 1);
        const int xrow2 = x.tok0 + n1 + static_cast<int>(rank) * (n2 >> 1);
        // both CTAs' copies; with FP8 weights the A slots are written by the
        // converter warps, whose arrivals the stage barrier counts instead
        const uint32_t bytes = 2 * ((kFp8 ? 0 : kABytes) + kBBytes + (n2 > 0 ? kBBytes : 0));
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&S->empty[stage], phase ^ 1u, abort_flag)) {
            failed = true;
            break;
          }
          const uint32_t lead_full = leader_addr(&S->full[stage]);
          uint8_t* st = s_stage0 + stage * C::kSlotBytes;
          if (rank == 0) mbar_arrive_expect_tx(&S->full[stage], bytes);
          if constexpr (kFp8) {
            // the code producer and the converters fill the A slot
          } else if (p.a_mn) {
            // K rows kb*64 .. +63 lie in packed tile k0 / a_tile_rows; M values
            // w0 .. w0+127 are its column blocks w0/64 and w0/64 + 1
            const int k0 = kb * BK;
            const int blk = (x.e * p.a_tiles + k0 / p.a_tile_rows) * p.a_mblocks + w0 / 64;
            tma_load_3d_pair(st, &tm_w, lead_full, 0, k0 % p.a_tile_rows, blk);
          } else if constexpr (kMode == kModeSwiGLU) {
            // the packed gate/up tile in quarter order (16 gate rows, then
            // their 16 up rows): 8 groups of 16 rows per block
            tma_load_4d_pair(st, &tm_w, lead_full, 0, 0, 0, (wblk + kb) * 8);
          } else {
            tma_load_3d_pair(st, &tm_w, lead_full, 0, wrow, wblk + kb);
          }
          uint8_t* sb = st + (kFp8 ? 0 : kABytes);  // B part 1, then part 2
          tma_load_2d_pair(sb, &tm_x, lead_full, kb * BK, xrow1);
          if (n2 > 0) tma_load_2d_pair(sb + kBBytes, &tm_x, lead_full, kb * BK, xrow2);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (failed) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (rank == 0 && lane == 0) {
      const int num_kb = p.K / BK;
      int stage = 0;
      uint32_t phase = 0;
      int astage = 0;  // FP8: A slot
      uint32_t asphase = 0;
      uint32_t aphase = 0;
      const uint32_t idesc0 = umma_idesc_bf16_f32_major(2 * kHalfRows, 16, p.a_mn != 0, false) & ~(0x3Fu << 17);
      int rs = 0;
      uint32_t rphase = 0;
      for (;;) {
        if (!wait_cluster(&S->rfull[rs], rphase, abort_flag)) {
          failed = true;
          break;
        }
        const int t = S->ring[rs];
        arrive_remote(leader_addr(&S->rempty[rs]));
        if (++rs == kRing) {
          rs = 0;
          rphase ^= 1u;
        }
        if (t < 0) break;
        const Tile x = decode(t, s_off, s_pre, p.E, p.m_tiles);
        const int n1 = min(x.n, kPartN), n2 = x.n - n1;
        const uint32_t idesc1 = idesc0 | (static_cast<uint32_t>(n1 >> 3) << 17);
        const uint32_t idesc2 = idesc0 | (static_cast<uint32_t>(max(n2, 16) >> 3) << 17);
        // the epilogue has drained the previous tile
        if (!wait_cluster(&S->tempty[0], aphase ^ 1u, abort_flag)) {
          failed = true;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base;
        for (int kb = 0; kb < num_kb; ++kb) {
          // FP8 weights: this CTA's A rows come with its converters'
          // arrivals, the peer's with its signaller's cluster release
          if (!mbar_wait(&S->full[stage], phase, abort_flag) ||
              (kFp8 && (!mbar_wait(&S->converted[astage], asphase, abort_flag) ||
                        (kb % C::kSigGroup == 0 && !wait_cluster(&S->apeer[astage], asphase, abort_flag))))) {
            failed = true;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a0 = kFp8 ? smem_addr(s_a0 + astage * kABytes) : smem_addr(s_stage0 + stage * kStageBytes);
          const uint32_t b1 = kFp8 ? smem_addr(s_stage0 + stage * C::kSlotBytes) : a0 + kABytes;
          // the stage's descriptors once; a K step of 16 advances the start
          // address (16-byte units) by 2 (K-major) or, for MN-major A, by
          // 16 rows of 128 bytes = 128
          const uint64_t da0 = p.a_mn ? sw128_mnmajor_desc(a0, kABytes / 2) : sw128_kmajor_desc(a0);
          const uint64_t da_step = p.a_mn ? (UMMA_K * 128) >> 4 : (UMMA_K * 2) >> 4;
          const uint64_t db1 = sw128_kmajor_desc(b1);
          const uint64_t db2 = db1 + (kBBytes >> 4);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            const uint64_t da = da0 + kk * da_step;
            const uint32_t accumulate = (kb | kk) != 0 ? 1u : 0u;
            umma_pair(d_tmem, da, db1 + 2 * kk, idesc1, accumulate);
            if (n2 > 0) umma_pair(d_tmem + kPartN, da, db2 + 2 * kk, idesc2, accumulate);
          }
          umma_commit_pair(&S->empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          if constexpr (kFp8) {
            umma_commit_pair(&S->aempty[astage]);
            if (++astage == C::kAStages) {
              astage = 0;
              asphase ^= 1u;
            }
          }
        }
        if (failed) break;
        umma_commit_pair(&S->tfull[0]);
        aphase ^= 1u;
      }
      umma_commit_pair(&S->drain);
    } else if (kFp8 && rank == 1 && lane == 0) {
      // ------------------------------------ FP8 signaller (peer CTA only)
      // per group of A slots: once this CTA's converter warps have written
      // their rows (their CTA-scope arrivals on `converted`), one
      // cluster-scope release arrive on the leader's apeer barrier of the
      // group's first slot makes the rows visible to the leader's MMA; the
      // converters never wait on that release themselves
      const int num_kb = p.K / BK;
      int astage = 0;
      uint32_t asphase = 0;
      int rs = 0;
      uint32_t rphase = 0;
      for (;;) {
        if (!wait_cluster(&S->rfull[rs], rphase, abort_flag)) {
          failed = true;
          break;
        }
        const int t = S->ring[rs];
        arrive_remote(leader_addr(&S->rempty[rs]));
        if (++rs == kRing) {
          rs = 0;
          rphase ^= 1u;
        }
        if (t < 0) break;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&S->converted[astage], asphase, abort_flag)) {
            failed = true;
            break;
          }
          // one release for the group's slots, on the group's first slot
          if (kb % C::kSigGroup == C::kSigGroup - 1)
            arrive_remote(leader_addr(&S->apeer[astage - (C::kSigGroup - 1)]));
          if (++astage == C::kAStages) {
            astage = 0;
            asphase ^= 1u;
          }
        }
        if (failed) break;
      }
    }
  } else if (kFp8 && warp >= 2 + kEpiWarps && warp < 2 + kEpiWarps + C::kConvWarps) {
    // ------------------------------------------------ FP8 code converters
    // thread = one 16-value piece (column c of the K block) of kRowsPer of
    // this CTA's 128 weight rows, kRowStep apart, per K block: its codes and
    // the piece's 16 scales from the code stage to bf16 in the MMA stage's A
    // slot, then a CTA-scope arrive on `converted`.  The rows of one thread
    // share their scales (same piece, same gate/up half) and their swizzle
    // offsets; a warp's code loads cover 8 whole 64-byte rows and its stores
    // 8 whole 128-byte rows, both free of bank conflicts.
    constexpr int kRowStep = 8 * (kFp8 ? C::kConvWarps : 4);
    constexpr int kRowsPer = kHalfRows / kRowStep;
    const int ci = (warp - 2 - kEpiWarps) * 32 + lane;
    const int c = ci & 3;
    const int rg = ci >> 2;
    // gate/up rows come in quarter order: 16 gate rows, then 16 up rows
    // (kRowStep is a multiple of 32, so every row of the thread is in the same half)
    const int half = (kMode == kModeSwiGLU) ? ((rg >> 4) & 1) : 0;
    const int code_off = rg * BK + ((c ^ ((rg >> 1) & 3)) << 4);
    const int a_off0 = rg * (BK * 2) + (((2 * c) ^ (rg & 7)) << 4);
    const int a_off1 = rg * (BK * 2) + (((2 * c + 1) ^ (rg & 7)) << 4);
    const int num_kb = p.K / BK;
    int astage = 0, cstage = 0;
    uint32_t asphase = 0, cphase = 0;
    int rs = 0;
    uint32_t rphase = 0;
    const uint32_t lead_rempty0 = leader_addr(&S->rempty[0]);
    for (;;) {
      if (!wait_cluster_warp(&S->rfull[rs], rphase, abort_flag)) {
        failed = true;
        break;
      }
      const int t = S->ring[rs];
      __syncwarp();
      if (lane == 0) arrive_remote(lead_rempty0 + rs * static_cast<uint32_t>(sizeof(uint64_t)));
      if (++rs == kRing) {
        rs = 0;
        rphase ^= 1u;
      }
      if (t < 0) break;
      for (int kb = 0; kb < num_kb; ++kb) {
        // the codes have landed: convert them into registers and free the
        // code stage, then wait until the MMA is done with the A slot, so
        // that only the stores, the fence and the arrive follow that wait
        if (!mbar_wait_warp(&S->cfull[cstage], cphase, abort_flag)) {
          failed = true;
          break;
        }
        const uint8_t* cs = s_code0 + cstage * C::kCodeStageBytes;
        const float* sc = reinterpret_cast<const float*>(cs + kCodeBytes) + half * 68 + 16 * c;
        float4 scl[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) scl[i] = *reinterpret_cast<const float4*>(sc + 4 * i);
        uint32_t o[kRowsPer][8];
#pragma unroll
        for (int j = 0; j < kRowsPer; ++j)
          convert_piece(*reinterpret_cast<const uint4*>(cs + code_off + j * kRowStep * BK), scl, o[j]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S->cempty[cstage]);
        if (!mbar_wait_warp(&S->aempty[astage], asphase ^ 1u, abort_flag)) {
          failed = true;
          break;
        }
        uint8_t* as = s_a0 + astage * kABytes;
#pragma unroll
        for (int j = 0; j < kRowsPer; ++j) {
          *reinterpret_cast<uint4*>(as + a_off0 + j * kRowStep * BK * 2) = make_uint4(o[j][0], o[j][1], o[j][2], o[j][3]);
          *reinterpret_cast<uint4*>(as + a_off1 + j * kRowStep * BK * 2) = make_uint4(o[j][4], o[j][5], o[j][6], o[j][7]);
        }
        // the generic-proxy stores become visible to the tensor cores' reads
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&S->converted[astage]);  // CTA scope: the leader's MMA thread or the peer's signaller
        if (++astage == C::kAStages) {
          astage = 0;
          asphase ^= 1u;
        }
        if (++cstage == C::kCodeStages) {
          cstage = 0;
          cphase ^= 1u;
        }
      }
      if (failed) break;
    }
  } else if (kFp8 && warp == 2 + kEpiWarps + C::kConvWarps) {
    // ----------------------------------------------- FP8 code producer
    // per K block: this CTA's 128 rows of codes (one 8 KB TMA box, 64-byte
    // swizzle) and the block's scale record, into the next code stage
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      const int num_kb = p.K / BK;
      const uint32_t rec_bytes = static_cast<uint32_t>(p.rec_floats) * 4u;
      int cstage = 0;
      uint32_t cphase = 0;
      int rs = 0;
      uint32_t rphase = 0;
      for (;;) {
        if (!wait_cluster(&S->rfull[rs], rphase, abort_flag)) {
          failed = true;
          break;
        }
        const int t = S->ring[rs];
        arrive_remote(leader_addr(&S->rempty[rs]));
        if (++rs == kRing) {
          rs = 0;
          rphase ^= 1u;
        }
        if (t < 0) break;
        const Tile x = decode(t, s_off, s_pre, p.E, p.m_tiles);
        const int ctile = x.mt * 2 + static_cast<int>(rank);  // this CTA's 128-row code tile
        const int64_t cblk = (static_cast<int64_t>(x.e) * p.code_tiles + ctile) * num_kb;
        const int64_t rec0 = (static_cast<int64_t>(x.e) * p.sc_tiles + (p.sc_per_cta ? ctile : x.mt)) * num_kb;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&S->cempty[cstage], cphase ^ 1u, abort_flag)) {
            failed = true;
            break;
          }
          uint8_t* cs = s_code0 + cstage * C::kCodeStageBytes;
          mbar_arrive_expect_tx(&S->cfull[cstage], kCodeBytes + rec_bytes);
          tma_load_2d(cs, &tm_w, &S->cfull[cstage], 0, static_cast<int32_t>((cblk + kb) * kHalfRows));
          bulk_load(cs + kCodeBytes, p.scales + (rec0 + kb) * p.rec_floats, rec_bytes, &S->cfull[cstage]);
          if (++cstage == C::kCodeStages) {
            cstage = 0;
            cphase ^= 1u;
          }
        }
        if (failed) break;
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int quad = warp & 3;            // TMEM lanes 32*quad .. +31
    const int part = (warp - 2) >> 2;     // which share of the tile's 32-token chunks
    const int ew = warp - 2;
    // one 2 KB buffer per warp: the staging of its stores
    uint8_t* tbuf = s_epi + ew * 2048;
    const uint32_t lead_tempty = leader_addr(&S->tempty[0]);
    uint32_t aphase = 0;
    int rs = 0;
    uint32_t rphase = 0;
    const uint32_t lead_rempty0 = leader_addr(&S->rempty[0]);
    for (;;) {
      if (!wait_cluster_warp(&S->rfull[rs], rphase, abort_flag)) {
        failed = true;
        break;
      }
      const int t = S->ring[rs];
      __syncwarp();
      if (lane == 0) arrive_remote(lead_rempty0 + rs * static_cast<uint32_t>(sizeof(uint64_t)));
      if (++rs == kRing) {
        rs = 0;
        rphase ^= 1u;
      }
      if (t < 0) break;
      const Tile x = decode(t, s_off, s_pre, p.E, p.m_tiles);
      if (!mbar_wait_warp_suspend(&S->tfull[0], aphase, abort_flag)) {
        failed = true;
        break;
      }
      tc_fence_after_sync();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
      // token columns 0 .. n-1 (TMEM columns 0..255 hold part 1, 256.. part 2)
      const int chunks = (x.n + 31) >> 5;
      const int per = (chunks + kEpiParts - 1) / kEpiParts;
      const int c_begin = part * per * 32;
      const int c_end = min((part + 1) * per * 32, x.n);
      // a, b hold chunk c (TMEM lanes 0-15 and 16-31 of the warp); the load
      // of chunk c + 32 is issued as soon as they have been consumed, so it
      // overlaps the stores of chunk c
      const uint32_t taddr_b = taddr + (16u << 16);
      // the accumulator goes back to the MMA as soon as the warp's last TMEM
      // load has landed, before that chunk's math and stores
      bool released = false;
      auto release = [&]() {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) arrive_remote_relaxed(lead_tempty);
        released = true;
      };
      uint32_t a[16], b[16];
      if (c_begin < c_end && kMode != kModeRows) {
        tmem_ld_16x256b_x4(taddr + c_begin, a);
        tmem_ld_16x256b_x4(taddr_b + c_begin, b);
        tmem_ld_wait();
      }
      if constexpr (kMode == kModeSwiGLU) {
        // The weight rows arrive in quarter order, so TMEM lanes 32q .. 32q+15
        // hold gate features j0 .. j0+15 (j0 = 64t + 16q of packed gate/up
        // tile t = 2*mt + rank) and lanes 32q+16 .. 32q+31 the up features of
        // the same j: a thread's registers of the two 16-lane loads pair up
        // element by element, and Silu(gate)*up needs no exchange.
        const int tp = x.mt * 2 + static_cast<int>(rank);
        __nv_bfloat16* hcol = p.out + static_cast<int64_t>(x.tok0) * p.out_cols + tp * 64 + quad * 16;
        // G,U for the backward: packed columns 128t + 16q (gate) and +64 (up)
        __nv_bfloat16* gucol =
            p.gu ? p.gu + static_cast<int64_t>(x.tok0) * 2 * p.out_cols + tp * 128 + quad * 16 : nullptr;
        // chunk c (in a, b): G,U stored if requested, then H as an stmatrix
        // fragment; the next chunk's TMEM loads are issued once a, b are read
        auto swiglu_chunk = [&](int c, uint32_t (&ph)[8]) {
          if (gucol != nullptr) {  // the raw pre-activations, for the backward
            uint32_t pk[16];
            pack_chunk(a, b, pk);
            stage_rows<4>(pk, tbuf, lane);
            rows_to_global_split(tbuf, lane, gucol + static_cast<int64_t>(c) * 2 * p.out_cols, 64, 2 * p.out_cols,
                                 x.valid - c);
          }
          float h[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) h[k] = silu_f32(__uint_as_float(a[k])) * __uint_as_float(b[k]);
          if (c + 32 < c_end) {
            tmem_ld_16x256b_x4(taddr + c + 32, a);
            tmem_ld_16x256b_x4(taddr_b + c + 32, b);
          }
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            ph[2 * g] = pack_bf16x2(h[4 * g], h[4 * g + 1]);
            ph[2 * g + 1] = pack_bf16x2(h[4 * g + 2], h[4 * g + 3]);
          }
        };
        // as in the row epilogue, the warp's last kHoldH chunks of H stay in
        // registers until the accumulator has been handed back
        const int n_chunks = c_begin < c_end ? (c_end - c_begin + 31) >> 5 : 0;
        const int n_stream = max(n_chunks - C::kHoldH, 0);
#pragma unroll 1
        for (int i = 0; i < n_stream; ++i) {
          const int c = c_begin + 32 * i;
          uint32_t ph[8];
          swiglu_chunk(c, ph);
          stage_rows_16f(ph, tbuf, lane);
          rows16f_to_global(tbuf, lane, hcol + static_cast<int64_t>(c) * p.out_cols, p.out_cols, x.valid - c);
          tmem_ld_wait();
        }
        uint32_t held[C::kHoldH][8];
#pragma unroll
        for (int hh = 0; hh < C::kHoldH; ++hh) {
          const int c = c_begin + 32 * (n_stream + hh);
          if (c < c_end) {
            if (c + 32 >= c_end) release();
            swiglu_chunk(c, held[hh]);
            if (c + 32 < c_end) tmem_ld_wait();
          }
        }
#pragma unroll
        for (int hh = 0; hh < C::kHoldH; ++hh) {
          const int c = c_begin + 32 * (n_stream + hh);
          if (c < c_end) {
            stage_rows_16f(held[hh], tbuf, lane);
            rows16f_to_global(tbuf, lane, hcol + static_cast<int64_t>(c) * p.out_cols, p.out_cols, x.valid - c);
          }
        }
      } else if constexpr (kMode == kModeSwiGLUBwd) {
        // lanes: features j0 .. j0+31 of dH (gate features of the packed
        // interleave: gate column (j / 64) * 128 + j % 64, up 64 further on)
        const int j0 = x.mt * 2 * kHalfRows + static_cast<int>(rank) * kHalfRows + quad * 32;
        const int64_t ld = 2 * static_cast<int64_t>(p.out_cols);
        const int64_t gcol0 = static_cast<int64_t>(j0 / 64) * 128 + j0 % 64;
        const __nv_bfloat16* gsrc = p.gu_in + static_cast<int64_t>(x.tok0) * ld + gcol0;
        __nv_bfloat16* gdst = p.out + static_cast<int64_t>(x.tok0) * ld + gcol0;
        // the accumulator before the row's gate, features j0 .. j0+31 of [P, f]
        __nv_bfloat16* hraw =
            p.dh_out ? p.dh_out + static_cast<int64_t>(x.tok0) * p.out_cols + j0 : nullptr;
        // G, U of the next 16 tokens are loaded into registers one half ahead,
        // so their latency overlaps the math and stores of the current half
        uint4 gv[2], uv[2];
        if (c_begin < c_end) {
          load_rows16(gv, lane, gsrc + static_cast<int64_t>(c_begin) * ld, ld, x.valid - c_begin);
          load_rows16(uv, lane, gsrc + static_cast<int64_t>(c_begin) * ld + 64, ld, x.valid - c_begin);
        }
#pragma unroll 1
        for (int c = c_begin; c < c_end; c += 32) {
          if (c + 32 >= c_end) release();
          // with row gates: lane i holds the gate of token column c + i
          const float gate_l =
              p.row_scale != nullptr && c + lane < x.valid ? __ldg(p.row_scale + x.tok0 + c + lane) : 1.0f;
          // two halves of 16 tokens (token groups 2h, 2h + 1) keep the
          // register footprint of G, U and the results small
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int r0 = c + 16 * h;
            uint32_t pg[8], pu[8], pr[8];
            store_rows16(tbuf, lane, gv);
            rows_to_fragment<2>(tbuf, lane, pg);
            store_rows16(tbuf, lane, uv);
            rows_to_fragment<2>(tbuf, lane, pu);
            // Silu(g) = g s, Silu'(g) = s (1 + g (1 - s)), s = sigmoid(g);
            // dG and dU replace G and U in pg, pu
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {
              // thread i's token columns in column group 2h + gg: 8(2h + gg) + 2(i % 4) and +1
              const float w0 = __shfl_sync(0xffffffffu, gate_l, 8 * (2 * h + gg) + 2 * (lane & 3));
              const float w1 = __shfl_sync(0xffffffffu, gate_l, 8 * (2 * h + gg) + 2 * (lane & 3) + 1);
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                const int i = 4 * (2 * h + gg) + 2 * (m & 1);
                const float r0v = __uint_as_float(m < 2 ? a[i] : b[i]);
                const float r1v = __uint_as_float(m < 2 ? a[i + 1] : b[i + 1]);
                pr[4 * gg + m] = pack_bf16x2(r0v, r1v);
                const float d0 = w0 * r0v;
                const float d1 = w1 * r1v;
                const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pg[4 * gg + m]));
                const float2 uf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pu[4 * gg + m]));
                const float s0 = sigmoid_f32(gf.x);
                const float s1 = sigmoid_f32(gf.y);
                pg[4 * gg + m] = pack_bf16x2(d0 * uf.x * s0 * (1.0f + gf.x * (1.0f - s0)),
                                             d1 * uf.y * s1 * (1.0f + gf.y * (1.0f - s1)));
                pu[4 * gg + m] = pack_bf16x2(d0 * gf.x * s0, d1 * gf.y * s1);
              }
            }
            if (h == 1 && c + 32 < c_end) {
              tmem_ld_16x256b_x4(taddr + c + 32, a);
              tmem_ld_16x256b_x4(taddr_b + c + 32, b);
            }
            const int rn = r0 + 16;  // the next half (of this chunk or the next)
            if (rn < c_end) {
              load_rows16(gv, lane, gsrc + static_cast<int64_t>(rn) * ld, ld, x.valid - rn);
              load_rows16(uv, lane, gsrc + static_cast<int64_t>(rn) * ld + 64, ld, x.valid - rn);
            }
            stage_rows<2>(pg, tbuf, lane);
            rows_to_global<16>(tbuf, lane, gdst + static_cast<int64_t>(r0) * ld, ld, x.valid - r0);
            stage_rows<2>(pu, tbuf, lane);
            rows_to_global<16>(tbuf, lane, gdst + static_cast<int64_t>(r0) * ld + 64, ld, x.valid - r0);
            if (hraw != nullptr) {
              stage_rows<2>(pr, tbuf, lane);
              rows_to_global<16>(tbuf, lane, hraw + static_cast<int64_t>(r0) * p.out_cols, p.out_cols, x.valid - r0);
            }
          }
          if (c + 32 < c_end) tmem_ld_wait();
        }
      } else {
        // lanes: output features i0 + lane; columns: tokens.  The warp's last
        // kHold chunks are read from TMEM into registers (as bf16 pairs)
        // before the accumulator goes back to the MMA, so that their staging
        // and stores overlap the next tile's MMAs; earlier chunks (tiles of
        // more than 2 * 32 * kHold tokens) are stored as they are read.
        const int i0 = x.mt * 2 * kHalfRows + static_cast<int>(rank) * kHalfRows + quad * 32;
        __nv_bfloat16* ycol = p.out + static_cast<int64_t>(x.tok0) * p.out_cols + i0;
        auto scale = [&](uint32_t (&v)[16], int c) {
          if (p.row_scale == nullptr) return;
          // lane i loads the gate of token column c + i; thread i's columns
          // are 8g + 2(i%4) and +1
          const float s_l = c + lane < x.valid ? __ldg(p.row_scale + x.tok0 + c + lane) : 1.0f;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const float s0 = __shfl_sync(0xffffffffu, s_l, 8 * g + 2 * (lane & 3));
            const float s1 = __shfl_sync(0xffffffffu, s_l, 8 * g + 2 * (lane & 3) + 1);
            v[4 * g] = __float_as_uint(s0 * __uint_as_float(v[4 * g]));
            v[4 * g + 1] = __float_as_uint(s1 * __uint_as_float(v[4 * g + 1]));
            v[4 * g + 2] = __float_as_uint(s0 * __uint_as_float(v[4 * g + 2]));
            v[4 * g + 3] = __float_as_uint(s1 * __uint_as_float(v[4 * g + 3]));
          }
        };
        // chunk c as a bf16 fragment (see pack_chunk): both 16-lane halves
        // read from TMEM behind one wait
        auto fill = [&](int c, uint32_t (&pk)[16]) {
          uint32_t v[16], w[16];
          tmem_ld_16x256b_x4(taddr + c, v);
          tmem_ld_16x256b_x4(taddr_b + c, w);
          tmem_ld_wait();
          scale(v, c);
          scale(w, c);
          pack_chunk(v, w, pk);
        };
        const int n_chunks = c_begin < c_end ? (c_end - c_begin + 31) >> 5 : 0;
        constexpr int kHold = C::kHold;
        const int n_stream = max(n_chunks - kHold, 0);
#pragma unroll 1
        for (int i = 0; i < n_stream; ++i) {
          const int c = c_begin + 32 * i;
          uint32_t pk[16];
          fill(c, pk);
          stage_rows<4>(pk, tbuf, lane);
          rows_to_global<32>(tbuf, lane, ycol + static_cast<int64_t>(c) * p.out_cols, p.out_cols, x.valid - c);
        }
        uint32_t held[kHold][16];
#pragma unroll
        for (int h = 0; h < kHold; ++h) {
          const int c = c_begin + 32 * (n_stream + h);
          if (c < c_end) fill(c, held[h]);
        }
        release();
#pragma unroll
        for (int h = 0; h < kHold; ++h) {
          const int c = c_begin + 32 * (n_stream + h);
          if (c < c_end) {
            stage_rows<4>(held[h], tbuf, lane);
            rows_to_global<32>(tbuf, lane, ycol + static_cast<int64_t>(c) * p.out_cols, p.out_cols, x.valid - c);
          }
        }
      }
      if (failed) break;
      if (!released) release();  // a warp without chunks in this tile
      aphase ^= 1u;
    }
  }

  if (failed && lane == 0) {
    record_status(p.status, kStatusTimeout);
    *abort_flag = 1;
  }
  // every MMA of the pair has completed once drain flips (the leader issued
  // them all); then let copies that a failed peer may still have in flight
  // land before the pair meets and frees its TMEM
  if (warp == 1) {
    if (lane == 0) {
      volatile int never = 0;
      mbar_wait(&S->drain, 0, &never);
    }
    __syncwarp();
  }
  __syncthreads();
  if (*abort_flag) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 10000000ull) __nanosleep(1000);
  }
  tc_fence_before_sync();
  cluster_sync();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

}  // namespace

bool grouped_gemm_2sm_supported(const GroupedGemmProblem& pb, Epilogue epi) {
  if (epi == Epilogue::kSwiGLU) return pb.out_cols % 128 == 0 && gate_up_half_tile(pb.out_cols) == 64;
  return pb.out_cols % 256 == 0 && down_tile_n(pb.out_cols) == 256;
}

namespace {

template <bool kFp8>
constexpr size_t smem_bytes(int E) {
  return 1024 + static_cast<size_t>(Cfg<kFp8>::kStages) * Cfg<kFp8>::kSlotBytes +
         static_cast<size_t>(Cfg<kFp8>::kAStages) * kABytes +
         static_cast<size_t>(Cfg<kFp8>::kCodeStages) * Cfg<kFp8>::kCodeStageBytes + kEpiBytes +
         sizeof(SmemT<kFp8>) + 2 * static_cast<size_t>(E + 1) * sizeof(int32_t);
}

// the largest expert count the library takes still fits the opt-in 227 KB
static_assert(smem_bytes<false>(MOE_MAX_EXPERTS) <= 227 * 1024, "shared memory of the paired GEMM");
static_assert(smem_bytes<true>(MOE_MAX_EXPERTS) <= 227 * 1024, "shared memory of the FP8-weight paired GEMM");
static_assert(Cfg<true>::kAStages % Cfg<true>::kSigGroup == 0 && (128 / BK) % Cfg<true>::kSigGroup == 0,
              "signal groups align with the A ring and with K blocks of a K % 128 == 0 problem");

template <bool kFp8>
cudaError_t launch_pairs(const CUtensorMap& mw, const CUtensorMap& mx, const Params& prm, int64_t P, int num_sms,
                         cudaStream_t stream) {
  const size_t smem = smem_bytes<kFp8>(prm.E);
  void (*kernel)(const CUtensorMap, const CUtensorMap, const Params);
  if constexpr (kFp8) {
    kernel = prm.mode == kModeSwiGLU ? grouped_gemm_2sm_kernel<kModeSwiGLU, true>
                                     : grouped_gemm_2sm_kernel<kModeRows, true>;
  } else {
    kernel = prm.mode == kModeSwiGLU      ? grouped_gemm_2sm_kernel<kModeSwiGLU, false>
             : prm.mode == kModeSwiGLUBwd ? grouped_gemm_2sm_kernel<kModeSwiGLUBwd, false>
                                          : grouped_gemm_2sm_kernel<kModeRows, false>;
  }
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  // persistent: one pair per two SMs, never more pairs than an upper bound on tiles
  const int64_t max_tiles = (P / kTileN + prm.E) * static_cast<int64_t>(prm.m_tiles);
  int pairs = num_sms / 2;
  if (max_tiles < pairs) pairs = static_cast<int>(max_tiles);
  kernel<<<2 * pairs, Cfg<kFp8>::kThreads, smem, stream>>>(mw, mx, prm);
  return cudaGetLastError();
}

Params base_params(const int32_t* offsets, int E, int K, int32_t* tile_counter, int32_t* status) {
  Params prm{};
  prm.static_tiles = g_static_tiles ? 1 : 0;
  prm.offsets = offsets;
  prm.status = status;
  prm.tile_counter = tile_counter;
  prm.E = E;
  prm.K = K;
  return prm;
}

}  // namespace

void set_static_tile_schedule(bool on) { g_static_tiles = on; }

cudaError_t launch_grouped_gemm_2sm(const GroupedGemmProblem& pb, Epilogue epi, int num_sms, cudaStream_t stream) {
  if (pb.P == 0) return cudaSuccess;
  if (!grouped_gemm_2sm_supported(pb, epi)) return cudaErrorNotSupported;
  const bool swiglu = epi == Epilogue::kSwiGLU;
  const int a_tile_rows = swiglu ? gate_up_tile_n(pb.out_cols) : down_tile_n(pb.out_cols);
  const int n_rows = pb.n_per_expert;  // weight rows per expert (2f or d)
  const int num_kb = pb.K / BK;
  CUtensorMap mw, mx;
  const int64_t blocks = static_cast<int64_t>(pb.E) * (n_rows / a_tile_rows) * num_kb;
  if (swiglu ? !make_bf16_map_gate_up_quads(&mw, pb.b, blocks)
             : !make_bf16_map_3d(&mw, pb.b, BK, a_tile_rows, blocks, BK, kHalfRows))
    return cudaErrorInvalidValue;
  if (!make_bf16_map_2d(&mx, pb.a, pb.P, pb.K, BK, kHalfRows)) return cudaErrorInvalidValue;
  Params prm = base_params(pb.offsets, pb.E, pb.K, pb.tile_counter, pb.status);
  prm.row_scale = swiglu ? nullptr : pb.row_scale;
  prm.out = static_cast<__nv_bfloat16*>(pb.out);
  prm.gu = swiglu ? static_cast<__nv_bfloat16*>(pb.gu_out) : nullptr;
  prm.m_tiles = n_rows / (2 * kHalfRows);
  prm.a_tile_rows = a_tile_rows;
  prm.a_tiles = n_rows / a_tile_rows;
  prm.out_cols = pb.out_cols;
  prm.mode = swiglu ? kModeSwiGLU : kModeRows;
  return launch_pairs<false>(mw, mx, prm, pb.P, num_sms, stream);
}

bool grouped_gemm_2sm_fp8_supported(const GroupedGemmProblem& pb, Epilogue epi) {
  if (!grouped_gemm_2sm_supported(pb, epi) || pb.K % 128 != 0 || pb.out_cols % 128 != 0) return false;
  // code rows (int32 TMA coordinates) of the whole projection
  return static_cast<int64_t>(pb.E) * pb.n_per_expert * (pb.K / BK) < (int64_t(1) << 31);
}

cudaError_t launch_grouped_gemm_2sm_fp8(const GroupedGemmProblem& pb, Epilogue epi, int num_sms,
                                        cudaStream_t stream) {
  if (pb.P == 0) return cudaSuccess;
  if (!grouped_gemm_2sm_fp8_supported(pb, epi) || pb.fp8_scales == nullptr) return cudaErrorNotSupported;
  const bool swiglu = epi == Epilogue::kSwiGLU;
  const int n_rows = pb.n_per_expert;  // weight rows per expert (2f or d)
  const int num_kb = pb.K / BK;
  CUtensorMap mw, mx;
  if (!make_u8_map_rows64_sw64(&mw, pb.b, static_cast<int64_t>(pb.E) * n_rows * num_kb, kHalfRows))
    return cudaErrorInvalidValue;
  if (!make_bf16_map_2d(&mx, pb.a, pb.P, pb.K, BK, kHalfRows)) return cudaErrorInvalidValue;
  Params prm = base_params(pb.offsets, pb.E, pb.K, pb.tile_counter, pb.status);
  prm.row_scale = swiglu ? nullptr : pb.row_scale;
  prm.out = static_cast<__nv_bfloat16*>(pb.out);
  prm.m_tiles = n_rows / (2 * kHalfRows);
  prm.a_tile_rows = kHalfRows;  // the producer's bf16 weight indexing is unused here, but kept defined
  prm.a_tiles = n_rows / kHalfRows;
  prm.out_cols = pb.out_cols;
  prm.mode = swiglu ? kModeSwiGLU : kModeRows;
  prm.scales = pb.fp8_scales;
  prm.code_tiles = n_rows / kHalfRows;
  // gate/up: a pair's two code tiles (gate/up features 128 mt .. +127) share
  // one 128-feature scale block; down: each CTA's 128 output features are one
  prm.sc_tiles = swiglu ? pb.out_cols / 128 : n_rows / kHalfRows;
  prm.sc_per_cta = swiglu ? 0 : 1;
  prm.rec_floats = swiglu ? kFp8GateUpRecord : kFp8DownRecord;
  return launch_pairs<true>(mw, mx, prm, pb.P, num_sms, stream);
}

bool dgrad_2sm_supported(const DgradProblem& g) {
  return g.m_out % (2 * kHalfRows) == 0 && g.K % BK == 0 && g.w_tile_rows % BK == 0 &&
         (g.mode != DgradEpilogue::kSwiGLUBwd || gate_up_half_tile(g.m_out) == 64);
}

cudaError_t launch_dgrad_2sm(const DgradProblem& g, int num_sms, cudaStream_t stream) {
  if (g.P == 0) return cudaSuccess;
  if (!dgrad_2sm_supported(g)) return cudaErrorNotSupported;
  CUtensorMap mw, mx;
  // packed weights as (64 columns, tile rows, blocks): two consecutive column
  // blocks of one packed tile per CTA and K block
  const int64_t blocks = static_cast<int64_t>(g.E) * g.w_tiles * (g.m_out / 64);
  if (!make_bf16_map_3d(&mw, g.w_packed, BK, g.w_tile_rows, blocks, BK, BK, 2)) return cudaErrorInvalidValue;
  if (!make_bf16_map_2d(&mx, g.tokens, g.P, g.K, BK, kHalfRows)) return cudaErrorInvalidValue;
  Params prm = base_params(g.offsets, g.E, g.K, g.tile_counter, g.status);
  prm.out = static_cast<__nv_bfloat16*>(g.out);
  prm.gu_in = static_cast<const __nv_bfloat16*>(g.gu_in);
  prm.m_tiles = g.m_out / (2 * kHalfRows);
  prm.a_tile_rows = g.w_tile_rows;
  prm.a_tiles = g.w_tiles;
  prm.a_mn = 1;
  prm.a_mblocks = g.m_out / 64;
  prm.out_cols = g.m_out;
  prm.mode = g.mode == DgradEpilogue::kSwiGLUBwd ? kModeSwiGLUBwd : kModeRows;
  if (g.mode == DgradEpilogue::kSwiGLUBwd) {
    prm.row_scale = g.row_scale;
    prm.dh_out = static_cast<__nv_bfloat16*>(g.dh_out);
  } else if (g.row_scale != nullptr || g.dh_out != nullptr) {
    return cudaErrorNotSupported;
  }
  return launch_pairs<false>(mw, mx, prm, g.P, num_sms, stream);
}

}  // namespace moe
