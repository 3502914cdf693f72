// Host-side declarations shared by the translation units of the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <cuda.h>
#include <cuda_runtime.h>

#include "moe_gb300.h"

namespace moe {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

// ---- stage 1 (hist: the per-chunk count table of stages 2-3, or null)
cudaError_t launch_route_topk(const float* logits, int64_t T, int E, int k, int n_groups, int renormalize,
                              int32_t* topk_idx, float* topk_w, int32_t* hist, int num_sms, cudaStream_t stream);

// ---- stage 1 with the router linear layer fused
int router_e_pad(int E);  // E rounded up to a multiple of 128
size_t router_smem_bytes(int E);
cudaError_t launch_pack_router(const void* w_router, int d, int E, void* packed, cudaStream_t stream);
cudaError_t launch_router_topk(const void* x, const void* w_packed, int64_t T, int d, int E, int k, int renormalize,
                               int32_t* topk_idx, float* topk_w, int32_t* hist, int32_t* status,
                               cudaStream_t stream);

// ---- backward of stage 5 and of the routing
// status (may be null) records a dest_row entry outside [0, T*k); such a
// slot is skipped (no row gradient, zero gate gradient).
cudaError_t launch_combine_backward(const void* dout, const void* mlp_out, const int32_t* dest_row, const float* w,
                                    int64_t T, int k, int d, void* d_mlp_out, float* d_w, int32_t* status,
                                    int num_sms, cudaStream_t stream);
cudaError_t launch_route_backward(const float* logits, const int32_t* idx, const float* d_w, int64_t T, int E, int k,
                                  int renormalize, float* d_logits, int num_sms, cudaStream_t stream);
// The output gradient on the expert rows when the expert outputs are not
// recomputed: plain[r] = dout[t] and, when gated is not null, gated[r] =
// bf16(w[t, j] * dout[t]) for the pair (t, j) at row r (dest_row); a row
// outside [0, T*k) is skipped and recorded in *status.
cudaError_t launch_dout_permute(const void* dout, const int32_t* dest_row, const float* w, int64_t T, int k, int d,
                                void* plain, void* gated, int32_t* status, int num_sms, cudaStream_t stream);
// The gate gradient from the down projection's input gradient before the
// gate: d_w[t*k + j] = <h[r], dh_raw[r]> (fp32) for the pair's row r; a row
// outside [0, T*k) gives 0 and is recorded in *status.  With w (the gates
// [T, k]) not null, each row of h is then replaced by bf16(w[t, j] h[r]).
cudaError_t launch_gate_grad(void* h, const void* dh_raw, const int32_t* dest_row, const float* w, int64_t T, int k,
                             int f, float* d_w, int32_t* status, int num_sms, cudaStream_t stream);

// ---- blockwise FP8 (E4M3) weights
cudaError_t launch_quantize_fp8(const void* w, int64_t n, uint8_t* codes, float* scales, int num_sms,
                                cudaStream_t stream);
cudaError_t launch_dequantize_fp8(const uint8_t* codes, const float* scales, int64_t n, void* out, int num_sms,
                                  cudaStream_t stream);
// The expert GEMMs' FP8 weight layout (moe_pack_weights_fp8): gate/up codes,
// down codes, gate/up scale records, down scale records; `offsets` (4
// entries, may be null) receives their byte offsets.  Needs d and f
// multiples of 128.
constexpr int kFp8GateUpRecord = 136;  // floats per gate/up scale record: 64 gate, 4 pad, 64 up, 4 pad
constexpr int kFp8DownRecord = 64;     // floats per down scale record
size_t fp8_packed_bytes(int E, int d, int f, size_t* offsets);
cudaError_t launch_pack_weights_fp8(const uint8_t* gate_codes, const float* gate_scales, const uint8_t* up_codes,
                                    const float* up_scales, const uint8_t* down_codes, const float* down_scales,
                                    int E, int d, int f, void* packed, int num_sms, cudaStream_t stream);

// ---- stages 2-3
constexpr int kDispatchThreads = 512;
constexpr int kDispatchPairsPerThread = 4;
constexpr int kDispatchChunk = kDispatchThreads * kDispatchPairsPerThread;  // pairs per block

inline int64_t dispatch_blocks(int64_t P) { return (P + kDispatchChunk - 1) / kDispatchChunk; }

// The per-chunk count table: hist[c][e] = pairs of chunk c (pairs
// 2048c .. 2048c + 2047) routed to expert e, int32, rows of
// dispatch_hist_stride(E) (E rounded up to 4) entries.
int dispatch_hist_stride(int E);
size_t dispatch_hist_bytes(int64_t P, int E);  // 256-byte aligned

// Writes every row of the table from topk_idx (no clearing needed).
cudaError_t launch_chunk_histogram(const int32_t* topk_idx, int64_t P, int E, int32_t* hist, int32_t* status,
                                   cudaStream_t stream);
// counts, offsets, dest_row, src_token and row_w (optional) from topk_idx and
// the complete table, one block per chunk and no block waiting on another.
cudaError_t launch_index(const int32_t* topk_idx, const float* topk_w, int64_t P, int E, int k, const int32_t* hist,
                         int32_t* counts, int32_t* offsets, int32_t* src_token, int32_t* dest_row, float* row_w,
                         int32_t* status, cudaStream_t stream);

// ---- stage 4 data movement and stage 5
// A dest_row entry outside [0, T*k) is skipped (no copy; no term of the sum)
// and recorded as MOE_ERR_BAD_INDEX in *status when status is not null.
cudaError_t launch_permute(const void* x, int64_t T, int d, const int32_t* dest_row, int k, void* x_perm,
                           int32_t* status, int num_sms, cudaStream_t stream);
cudaError_t launch_combine(const void* y, const int32_t* dest_row, const float* topk_w, int64_t T, int k, int d,
                           void* out, int32_t* status, int num_sms, cudaStream_t stream);

// ---- weights
int gate_up_half_tile(int f);  // N columns of gate (and of up) in one GEMM tile
int gate_up_tile_n(int f);     // N rows of one packed gate/up weight tile (2 * half tile)
int down_tile_n(int d);        // N rows of one packed down weight tile (256, 128 or 64)
cudaError_t launch_pack_weights(const void* w_gate, const void* w_up, const void* w_down, int E, int d, int f,
                                void* packed, cudaStream_t stream);

// ---- stage 4 expert GEMMs
struct GroupedGemmProblem {
  const void* a;           // [P, K] bf16 (x_perm or h); with gather_rows: [a_rows, K] (x)
  const void* b;           // packed weights of this projection, [E * n_per_expert, K] bf16
  const int32_t* offsets;  // [E+1]
  const float* row_scale;  // [P] or null (down projection only)
  void* out;               // [P, out_cols] bf16
  int64_t P;
  int E;
  int K;
  int n_per_expert;        // 2f (gate/up) or d (down)
  int out_cols;            // f or d
  int32_t* tile_counter;   // zeroed before launch
  int32_t* status;
  const int32_t* gather_rows = nullptr;  // gate/up only: A row r is a[gather_rows[r]] (src_token)
  void* gu_out = nullptr;                // gate/up, paired form only: also store G, U [P, 2f]
  int64_t a_rows = 0;                    // rows of a when gathering (T)
  const float* fp8_scales = nullptr;     // FP8 weights: b holds codes, these the scale records
};
enum class Epilogue { kSwiGLU, kScale };
cudaError_t launch_grouped_gemm(const GroupedGemmProblem& pb, Epilogue epi, int num_sms, cudaStream_t stream);
// The paired-SM form (weights as the 256-row operand, up to 512 of an
// expert's tokens as N): used by launch_grouped_gemm when the weight rows
// per expert (2f, or d) are a multiple of 256.
// The paired GEMMs' tile schedule for the rest of the process: a shared
// atomic counter (default) or a static stride over the pairs (measurement).
void set_static_tile_schedule(bool on);
// A kernel holding n_sms SMs (one block each) for duration_ns.
cudaError_t launch_occupy(int n_sms, uint64_t duration_ns, cudaStream_t stream);
bool grouped_gemm_2sm_supported(const GroupedGemmProblem& pb, Epilogue epi);
cudaError_t launch_grouped_gemm_2sm(const GroupedGemmProblem& pb, Epilogue epi, int num_sms, cudaStream_t stream);
// The paired form reading FP8 weights (moe_pack_weights_fp8's layout): b =
// this projection's codes, fp8_scales = its scale records.  Converter warps
// dequantise each K block in shared memory exactly as
// moe_dequantize_fp8_blockwise does, so the results equal the bf16 path's on
// those dequantised weights bit for bit.  Needs what the paired form needs
// and d, f multiples of 128.
bool grouped_gemm_2sm_fp8_supported(const GroupedGemmProblem& pb, Epilogue epi);
cudaError_t launch_grouped_gemm_2sm_fp8(const GroupedGemmProblem& pb, Epilogue epi, int num_sms,
                                        cudaStream_t stream);

// A dgrad GEMM of the backward on SM pairs: out[r, :] = tokens[r, :] W_e^T
// for the rows r of expert e, with W_e the forward's packed weights read
// transposed (the M = m_out output features run along a packed tile's
// columns, K along its rows).
enum class DgradEpilogue { kRows, kSwiGLUBwd };
struct DgradProblem {
  const void* tokens;      // [P, K] bf16: [dG | dU] interleaved (K = 2f) or dY (K = d)
  const void* w_packed;    // packed gate/up (tile rows 128 along 2f) or down (tile rows 256 along d)
  const int32_t* offsets;  // [E+1]
  int64_t P;
  int E;
  int K;
  int m_out;               // d (dX) or f (dH)
  int w_tile_rows;         // rows of one packed tile
  int w_tiles;             // packed tiles per expert (= K / w_tile_rows)
  DgradEpilogue mode;      // kRows: out = dX [P, d]; kSwiGLUBwd: out = dG,dU [P, 2f] from gu_in
  const void* gu_in;       // kSwiGLUBwd: the saved G, U [P, 2f]
  void* out;
  int32_t* tile_counter;
  int32_t* status;
  // kSwiGLUBwd only, both optional: the gate of each row, applied to the
  // accumulator before dG, dU are formed (the tokens are then the ungated
  // output gradient), and [P, f] bf16 receiving the accumulator as it is
  const float* row_scale = nullptr;
  void* dh_out = nullptr;
};
bool dgrad_2sm_supported(const DgradProblem& g);
cudaError_t launch_dgrad_2sm(const DgradProblem& g, int num_sms, cudaStream_t stream);

// ---- stage 4 backward: expert GEMMs of the backward pass
struct BackwardGemmArgs {
  int64_t P;
  int E, d, f;
  const int32_t* offsets;  // [E+1]
  const void* w_gate_up;   // packed gate/up weights (first part of moe_pack_weights' output)
  const void* w_down;      // packed down weights (second part)
  const void* x_perm;      // [P, d]
  const void* dy;          // [P, d] gradient of the expert outputs
  void* h;                 // [P, f]   (written by the gate/up GEMM, read by the down wgrad)
  void* gu;                // [P, 2f]  gate and up pre-activations, interleaved per gate/up tile
  void* dgu;               // [P, 2f]  their gradients, same order
  void* dx_perm;           // [P, d]
  void* dw_gate;           // [E, d, f] or null (skip both gate/up weight gradients)
  void* dw_up;             // [E, d, f]
  void* dw_down;           // [E, f, d] or null
  int32_t* counters;       // the workspace header's 6 tile counters, zeroed before launch:
                           // [0] gate/up (save), [2..5] dgrad down, dgrad gate/up,
                           // wgrad down, wgrad gate/up
  int32_t* status;
  // Optional (the layer backward without the recomputed down projection;
  // needs backward_gate_grad_in_dgrad): the dgrad down GEMM then takes the
  // ungated output gradient rows dy_dgrad, applies each row's gate row_w to
  // its accumulator and writes that accumulator before the gate to dh_raw
  // [P, f]; dy stays the gated rows for the down weight gradient.
  const void* dy_dgrad;
  const float* row_w;
  void* dh_raw;
  // Optional operands of the down weight gradient in place of h and dy
  // (its result H^T dY equals (gated H)^T (ungated rows)).
  const void* h_wgrad;
  const void* dy_wgrad;
};
// Whether the dgrad down GEMM of this shape runs on SM pairs, where it can
// take row gates and write dh_raw (BackwardGemmArgs).
bool backward_gate_grad_in_dgrad(int E, int d, int f);
// Gate/up GEMM that writes H and, for the backward, G and U.
cudaError_t launch_gate_up_save(const BackwardGemmArgs& a, int num_sms, cudaStream_t stream);
// dG,dU (from dY, G, U), dX, and the weight gradients, in that order;
// events[0..3] (optional) are recorded after each of the four GEMMs.
cudaError_t launch_swiglu_backward_gemms(const BackwardGemmArgs& a, int num_sms, cudaStream_t stream,
                                         void* const* events);
// The same in two halves: dG,dU then dX (events[0..1] after each), and the
// down then the gate/up weight gradients (events[0..1] after each).
cudaError_t launch_backward_dgrad_gemms(const BackwardGemmArgs& a, int num_sms, cudaStream_t stream,
                                        void* const* events);
cudaError_t launch_backward_wgrad_gemms(const BackwardGemmArgs& a, int num_sms, cudaStream_t stream,
                                        void* const* events);

// Tiled bf16 TMA maps, 128-byte swizzle, zero fill outside the tensor.
// 2-D: row-major [rows, cols], box [box_rows, box_cols].  3-D: dense
// [d2][d1][d0] (d0 contiguous), box [1][box1][box0].
bool make_bf16_map_2d(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_cols, int box_rows);
bool make_bf16_map_3d(CUtensorMap* map, const void* ptr, int64_t d0, int64_t d1, int64_t d2, int box0, int box1,
                      int box2 = 1);
bool make_bf16_map_2d_sw64(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_cols,
                           int box_rows);
bool make_bf16_map_gate_up_quads(CUtensorMap* map, const void* ptr, int64_t blocks);
bool make_bf16_map_col_blocks(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_rows,
                              int box_blocks);
// Byte rows of 64 (FP8 codes) as [rows][64], box of box_rows rows, 64-byte
// swizzle: 16-byte piece c of row r lands at piece c ^ ((r >> 1) & 3).
bool make_u8_map_rows64_sw64(CUtensorMap* map, const void* ptr, int64_t rows, int box_rows);

// Bounded-wait check: one block waits on a phase that never completes and
// records a timeout in *status after limit_ns.
cudaError_t launch_wait_timeout(int32_t* status, uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_activation(const float* z, int64_t n, float* silu, float* sigmoid, int num_sms,
                              cudaStream_t stream);

// Device properties of the current device (cached per device).
struct DeviceInfo {
  int device;
  int num_sms;
  int cc_major, cc_minor;
};
cudaError_t current_device_info(DeviceInfo* info);

// Sets the text moe_last_error returns on the calling host thread.
void set_last_error(const std::string& msg);

// Host checks of the routing sizes every routing entry point shares: T >= 0,
// 1 <= E <= MOE_MAX_EXPERTS, 1 <= k <= min(E, MOE_MAX_TOPK), T*k < 2^31.
// Sets the last-error text on failure.
moe_status_t check_routing(int64_t T, int32_t E, int32_t k);

}  // namespace moe
