/*
 * moe_gb300.h — C ABI of the single-GPU Mixture-of-Experts layer, forward
 * and backward (GB300, sm_103a).
 *
 * The layer follows "Scalable Pretraining of Large MoE LMs on Aurora Super
 * Computer", §3.1 FastSparseMoE, Algorithm 1 (FastSparseMoEBlock), on one
 * device without expert parallelism:
 *   stage 1  Softmax and TopK of the router logits        -> moe_route_topk
 *   stage 2  per-expert token counts and prefix sums      -> moe_dispatch_scan
 *   stage 3  index generation (row->token, pair->row)     -> moe_dispatch_scan
 *   stage 4  mlp_in = input[input_indices]                -> moe_permute
 *            grouped gate/up GEMMs, Silu(gate)*up, grouped
 *            down GEMM                                    -> moe_grouped_swiglu
 *   stage 5  output reduction weighted by the TopK weights -> moe_combine
 * and moe_forward runs all of them (moe_forward_gathered without the
 * permuted copy; moe_forward_routed from the tokens and the router weights;
 * moe_forward_host / moe_forward_host_stream from host buffers).  The
 * backward: stage 5 -> moe_combine_backward, stage 1 -> moe_route_backward,
 * stage 4 -> moe_grouped_gate_up_save + moe_grouped_swiglu_backward, and
 * moe_backward runs the whole layer backward with the forward recomputed.
 * Sizes follow the problem statement of that section: T tokens of hidden
 * size d, E routed experts, top-k, expert hidden size f; P = T*k routed
 * (token, slot) pairs.
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE memory owned by the caller unless a parameter says
 *     "host".  Nothing is allocated by the library; scratch comes from a
 *     caller-provided workspace sized by the matching *_workspace_bytes query
 *     and must be 256-byte aligned.
 *   - Tensors are dense and row-major.  "bf16" buffers hold IEEE bfloat16
 *     bit patterns (2 bytes each); they are typed void* here.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and returns without waiting for it.  Only
 *     moe_read_device_status, moe_get_device_status,
 *     moe_dispatch_noalloc_status, moe_forward_host and
 *     moe_forward_host_stream synchronise.
 *   - Argument errors are found on the host and returned at once with no
 *     work enqueued.  Errors found by a kernel (a bounded wait that ran out,
 *     an out-of-range expert index or row index) are written to a status
 *     word at the start of the workspace and read back with
 *     moe_get_device_status or moe_read_device_status.
 *   - Calls that share a workspace must not overlap on the GPU.
 *   - Supported sizes: 1 <= E <= 1024, 1 <= k <= min(E, 32), 0 <= T,
 *     T*k < 2^31.  The GEMM stages and moe_forward need d and f to be
 *     multiples of 64 in [64, 65536] (whole 128-byte K blocks for the
 *     tensor cores); moe_permute and moe_combine need d % 8 == 0 (16-byte
 *     rows).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_GB300_ABI_VERSION 1
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOPK 32

typedef void* moe_stream_t; /* cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* NULL pointer, negative or inconsistent size   */
  MOE_ERR_UNSUPPORTED = 2,   /* size outside the supported range above        */
  MOE_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed   */
  MOE_ERR_TIMEOUT = 4,       /* a kernel's bounded wait ran out (device)      */
  MOE_ERR_BAD_INDEX = 5,     /* an expert index outside [0, E) (device)       */
  MOE_ERR_WORKSPACE = 6,     /* workspace NULL, misaligned or too small       */
  MOE_ERR_NO_DEVICE = 7      /* no CUDA device, or not an sm_103 device       */
} moe_status_t;

/* ABI version of the loaded library (MOE_GB300_ABI_VERSION). */
MOE_API int moe_abi_version(void);

/* Static text for a status code. */
MOE_API const char* moe_status_string(moe_status_t status);

/* Text describing the last error returned on the calling host thread
 * (thread-local; valid until the next call on that thread). */
MOE_API const char* moe_last_error(void);

/* ------------------------------------------------------------------------
 * Stage 1 — router Softmax and TopK (Algorithm 1, stage 1).
 *   logits    [T, E] fp32, one row per token.
 *   topk_idx  [T, k] int32 out: slot j holds the (j+1)-th largest logit;
 *             ties go to the smaller expert index, -0.0 equals +0.0.
 *   topk_w    [T, k] fp32 out: softmax probability of that expert; when
 *             renormalize != 0, divided by the sum over the k selected
 *             (equal to the softmax over the k selected logits).
 * Logits must be finite.  T == 0 enqueues nothing.
 * Errors: MOE_ERR_INVALID_ARG (NULL with T > 0, T < 0),
 *         MOE_ERR_UNSUPPORTED (E or k out of range), MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_route_topk(const float* logits, int64_t T, int32_t E, int32_t k,
                            int32_t renormalize, int32_t* topk_idx, float* topk_w,
                            moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 1 with group-limited routing ("Training a 1T-Params MoE on EU
 * public infrastructure", Group-limited expert routing): the E experts are
 * split into n_groups groups of consecutive indices, [g*E/G, (g+1)*E/G),
 * and each token takes exactly k/G experts from every group (its best ones
 * inside the group, same order and ties as moe_route_topk), so every group
 * receives exactly T*k/G pairs.  Slots hold the k selected experts in
 * descending logit order; gates as in moe_route_topk (softmax over all E,
 * renormalised over the selected k when renormalize != 0).
 * n_groups = 1 is moe_route_topk.
 * Errors: as moe_route_topk, and MOE_ERR_UNSUPPORTED when n_groups < 1 or
 * does not divide both E and k.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_route_topk_grouped(const float* logits, int64_t T, int32_t E, int32_t k,
                                    int32_t n_groups, int32_t renormalize,
                                    int32_t* topk_idx, float* topk_w, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 1 with the router linear layer fused (Algorithm 1, stage 1:
 * logits = Router(input); Softmax; TopK): the logits x @ w_router of a
 * 128-token tile are accumulated on the tensor cores (bf16 operands, fp32
 * accumulation) and reduced to the top-k in the same kernel, without being
 * written to memory.  Selection order, ties and gates as moe_route_topk,
 * applied to those fp32 logits.
 *   w_router  [d, E] bf16, packed once by moe_pack_router_weights into
 *             moe_router_packed_bytes(d, E) bytes (K-major, E padded with
 *             zero columns to a multiple of 128);
 *   x         [T, d] bf16; topk_idx [T, k] int32 out; topk_w [T, k] fp32 out;
 *   workspace 256 bytes (status word).
 * Supported: E <= 512, d a multiple of 64 in [64, 65536], k <= min(E, 32).
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE,
 *         MOE_ERR_NO_DEVICE, MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
MOE_API size_t moe_router_packed_bytes(int32_t d, int32_t E);
MOE_API moe_status_t moe_pack_router_weights(const void* w_router, int32_t d, int32_t E, void* packed,
                                     moe_stream_t stream);
MOE_API moe_status_t moe_router_topk(const void* x, const void* router_packed, int64_t T, int32_t d,
                             int32_t E, int32_t k, int32_t renormalize,
                             int32_t* topk_idx, float* topk_w,
                             void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Stages 2 and 3 — token counts, group boundaries and index generation
 * (Algorithm 1, stages 2-3), as one stable counting sort of the P pairs
 * p = t*k + j by expert:
 *   counts    [E] int32 out: pairs routed to each expert (token counts).
 *   offsets   [E+1] int32 out: exclusive prefix sum of counts, offsets[E]=P
 *             (cumulative token counts: expert e owns rows
 *             [offsets[e], offsets[e+1])).
 *   dest_row  [P] int32 out: row of pair p (output indices) =
 *             offsets[e] + number of pairs q < p routed to the same expert;
 *             rows of one expert are therefore in ascending token order.
 *   src_token [P] int32 out: token of the pair placed at each row (input
 *             indices); src_token[dest_row[p]] == p / k.
 *   row_w     [P] fp32 out, optional (NULL skips it): row_w[dest_row[p]] =
 *             topk_w[p]; needs topk_w.
 *   topk_idx  [T, k] int32 in; topk_w [T, k] fp32 in, optional.
 * Implementation: a table of per-chunk expert counts (chunks of 2,048
 * pairs), then one pass, a block per chunk, that takes every chunk's
 * per-expert base from the table's column sums; no block waits on another.
 * An expert index outside [0, E) sets MOE_ERR_BAD_INDEX in the device
 * status word and its pair is dropped (dest_row = -1).
 * Workspace: moe_dispatch_workspace_bytes(T, E, k) bytes.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE,
 *         MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
MOE_API size_t moe_dispatch_workspace_bytes(int64_t T, int32_t E, int32_t k);
MOE_API moe_status_t moe_dispatch_scan(const int32_t* topk_idx, const float* topk_w,
                               int64_t T, int32_t E, int32_t k,
                               int32_t* counts, int32_t* offsets,
                               int32_t* src_token, int32_t* dest_row, float* row_w,
                               void* workspace, size_t workspace_bytes,
                               moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_dispatch_scan_noalloc — the same counts, offsets and index maps as
 * moe_dispatch_scan, for callers that cannot allocate device memory at
 * call time: plugins and framework extensions that receive only their
 * input and output buffers, and latency-critical loops that must not call
 * cudaMalloc.  The pages have no counterpart of this entry point.
 *   Arguments and outputs are those of moe_dispatch_scan, without the
 *   workspace.  The scratch (status word and count table) is a fixed 4 MiB
 *   device array inside the library (held on every GPU that loads it until the process exits):
 *   problems whose scratch, moe_dispatch_workspace_bytes(T, E, k), exceeds
 *   4 MiB are rejected with MOE_ERR_UNSUPPORTED (for example E = 384 and
 *   k = 8 fit up to about 699,000 tokens).
 *   The first call on a device looks up the array's address with that
 *   device current; make it before any stream capture.  All calls share
 *   the array: calls that overlap on the GPU race and must be serialised
 *   by the caller.  Allocates nothing (no cudaMalloc, cudaFree or
 *   allocating library routine).  A pair with an out-of-range expert index
 *   gets dest_row = -1, as with moe_dispatch_scan.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_NO_DEVICE,
 *         MOE_ERR_CUDA.
 *
 * moe_dispatch_noalloc_status waits for `stream` and copies into *status
 * (host memory) the device status of the latest moe_dispatch_scan_noalloc
 * on the current device: MOE_OK, or MOE_ERR_BAD_INDEX when an expert index
 * was outside [0, E).  The next call clears it, so read
 * it before that call is enqueued.  Allocates nothing.
 * Errors: MOE_ERR_INVALID_ARG (NULL status), MOE_ERR_NO_DEVICE, MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_dispatch_scan_noalloc(const int32_t* topk_idx, const float* topk_w,
                                       int64_t T, int32_t E, int32_t k,
                                       int32_t* counts, int32_t* offsets,
                                       int32_t* src_token, int32_t* dest_row, float* row_w,
                                       moe_stream_t stream);
MOE_API moe_status_t moe_dispatch_noalloc_status(moe_stream_t stream, int32_t* status);

/* ------------------------------------------------------------------------
 * Stage 4, first step — mlp_in = input[input_indices] (Algorithm 1,
 * stage 4), done from the token side: each token row of x is read once and
 * written to its k rows, x_perm[dest_row[t*k + j]] = x[t].  The result is
 * the same as gathering x_perm[r] = x[src_token[r]].
 *   x [T, d] bf16 in; dest_row [T*k] int32 in (a bijection onto [0, T*k));
 *   x_perm [T*k, d] bf16 out.
 * An entry of dest_row outside [0, T*k) (such as the -1 the dispatch pass
 * writes for a pair it could not place) is skipped: nothing is written for
 * that pair, and no memory outside x_perm is touched.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_permute(const void* x, int64_t T, int32_t d, const int32_t* dest_row,
                         int32_t k, void* x_perm, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Expert weights in the layout the grouped GEMM reads.  Algorithm 1,
 * stage 4 concatenates the per-expert weights of one projection into one
 * tensor; this call does that once, ahead of the forward (it is a layout
 * transform, not part of the per-step path):
 *   w_gate, w_up [E, d, f] bf16 in (gate = x @ w_gate[e]);
 *   w_down       [E, f, d] bf16 in (y = h @ w_down[e]);
 *   packed       moe_packed_weight_bytes(E, d, f) bytes out (3*E*d*f bf16):
 *                the gate/up projection, then the down projection, each
 *                stored K-major and tile-major: element (e, n, k) of a
 *                projection with N tile BN and K = 64 * nkb sits at
 *                (((e * N/BN + n/BN) * nkb + k/64) * BN + n%BN) * 64 + k%64,
 *                so that one GEMM stage's weights are one contiguous block.
 *                Gate/up: N = 2f, K = d, BN = 128, and N tile t holds
 *                gate columns 64t .. 64t+63 then the same up columns.
 *                Down: N = d, K = f, BN = 256, 128 or 64, the largest
 *                dividing d.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
MOE_API size_t moe_packed_weight_bytes(int32_t E, int32_t d, int32_t f);
MOE_API moe_status_t moe_pack_weights(const void* w_gate, const void* w_up, const void* w_down,
                              int32_t E, int32_t d, int32_t f, void* packed,
                              moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Blockwise FP8 expert weights ("Training a 1T-Params MoE on EU public
 * infrastructure", FP8 expert weight all-gather): the n values of a weight
 * tensor are cut into blocks of 128 consecutive values; each block gets one
 * fp32 scale = amax / 448 (1 for an all-zero block) and its values become
 * E4M3 codes of w / scale (fp32 division, round to nearest even, saturating
 * at +-448).  Dequantisation gives bf16(E4M3 value * scale), the weights
 * the expert computation then uses (pack them with moe_pack_weights); per
 * value the error is at most ~6% of its block's maximum.
 *   w [n] bf16; codes [n] uint8 (E4M3 bit patterns); scales [n/128] fp32.
 * n must be a multiple of 128.  Errors: MOE_ERR_INVALID_ARG,
 * MOE_ERR_NO_DEVICE, MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_quantize_fp8_blockwise(const void* w, int64_t n, uint8_t* codes, float* scales,
                                        moe_stream_t stream);
MOE_API moe_status_t moe_dequantize_fp8_blockwise(const uint8_t* codes, const float* scales, int64_t n,
                                          void* w_out, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * FP8 expert weights read by the expert GEMMs themselves ("Training a
 * 1T-Params MoE on EU public infrastructure", FP8 expert weight all-gather:
 * the weights travel as E4M3 codes with one fp32 scale per 128 values and
 * become bf16 before the expert computation).  moe_pack_weights_fp8 lays out
 * the codes and scales of the three projections, as
 * moe_quantize_fp8_blockwise produced them, for the FP8-weight GEMMs:
 *   gate_codes, up_codes [E, d, f] uint8 and down_codes [E, f, d] uint8 (the
 *   stored weights' order); gate_scales, up_scales [E*d*f/128] and
 *   down_scales [E*f*d/128] fp32 (one per 128 consecutive stored values);
 *   packed  moe_fp8_packed_weight_bytes(E, d, f) bytes out (about half of
 *           moe_packed_weight_bytes): the codes of each projection in
 *           128-row tiles of 64-value K blocks (8 KB each; gate/up tile t
 *           holds gate features 64t .. 64t+63 and the same up features,
 *           16 gate rows then their 16 up rows, down tile t output features
 *           128t .. 128t+127), then per (expert, 128-feature block, K block)
 *           a record of that block's 64 scales of each projection.
 * moe_forward_fp8 is moe_forward with those weights: each GEMM stage's codes
 * are dequantised in shared memory to bf16(E4M3 value x scale), the product
 * rounded once in fp32 -- exactly what moe_dequantize_fp8_blockwise gives --
 * and the tensor cores run on them as on bf16 weights, so every
 * intermediate and the output equal moe_forward's on the dequantised,
 * moe_pack_weights-packed weights bit for bit.  The HBM traffic of the
 * weights is halved.  Arguments, workspace, layout and errors as
 * moe_forward; moe_forward_fp8_timed records events as moe_forward_timed.
 * Codes must be finite (as the quantiser writes them).
 * Supported: d and f multiples of 128 (the forward: d a multiple of 256).
 * Errors: MOE_ERR_INVALID_ARG (NULL, misaligned: codes 16-byte, packed
 *         256-byte), MOE_ERR_UNSUPPORTED, MOE_ERR_NO_DEVICE, MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
MOE_API size_t moe_fp8_packed_weight_bytes(int32_t E, int32_t d, int32_t f);
MOE_API moe_status_t moe_pack_weights_fp8(const uint8_t* gate_codes, const float* gate_scales,
                                          const uint8_t* up_codes, const float* up_scales,
                                          const uint8_t* down_codes, const float* down_scales, int32_t E,
                                          int32_t d, int32_t f, void* packed, moe_stream_t stream);
MOE_API moe_status_t moe_forward_fp8(const void* x, const float* logits, const void* packed_fp8, int64_t T,
                                     int32_t d, int32_t E, int32_t k, int32_t f, int32_t renormalize, void* out,
                                     int32_t* topk_idx_out, float* topk_w_out, void* workspace,
                                     size_t workspace_bytes, moe_stream_t stream);
MOE_API moe_status_t moe_forward_fp8_timed(const void* x, const float* logits, const void* packed_fp8, int64_t T,
                                           int32_t d, int32_t E, int32_t k, int32_t f, int32_t renormalize,
                                           void* out, void* workspace, size_t workspace_bytes,
                                           moe_stream_t stream, void* const* events);

/* ------------------------------------------------------------------------
 * Stage 4, expert computation — the grouped gate/up GEMM with
 * Silu(gate)*up and the grouped down GEMM (Algorithm 1, stage 4), over the
 * expert groups given by offsets, on the tensor cores (bf16 operands, fp32
 * accumulation):
 *   h[r, :] = bf16( silu(x_perm[r] @ Wg[e]) * (x_perm[r] @ Wu[e]) )
 *   y[r, :] = bf16( row_scale[r] * (h[r] @ Wd[e]) )   (scale 1 if NULL)
 * for every row r in [offsets[e], offsets[e+1]).
 *   x_perm [P, d] bf16 in; offsets [E+1] int32 in (offsets[E] == P, as
 *   moe_dispatch_scan writes it); packed from moe_pack_weights;
 *   row_scale [P] fp32 in, optional (the gate of each row, row_w);
 *   h [P, f] bf16 out; y [P, d] bf16 out.
 * Experts with no rows cost nothing.  Tiles are handed to persistent
 * blocks from an atomic counter.
 * Workspace: moe_grouped_swiglu_workspace_bytes() bytes.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE,
 *         MOE_ERR_NO_DEVICE, MOE_ERR_CUDA; MOE_ERR_TIMEOUT in the status word.
 * ---------------------------------------------------------------------- */
MOE_API size_t moe_grouped_swiglu_workspace_bytes(void);
MOE_API moe_status_t moe_grouped_swiglu(const void* x_perm, const int32_t* offsets, int64_t P,
                                int32_t E, int32_t d, int32_t f, const void* packed,
                                const float* row_scale, void* h, void* y,
                                void* workspace, size_t workspace_bytes,
                                moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 5 — output reduction, forward (Algorithm 1, stage 5):
 *   out[t, :] = bf16( sum_{j<k} w[t, j] * y[dest_row[t*k + j], :] )
 * summed in fp32 in slot order; w = topk_w, or 1 when topk_w is NULL (the
 * rows already carry their gate, as moe_grouped_swiglu writes them with
 * row_scale).
 *   y [T*k, d] bf16 in; dest_row [T*k] int32 in; topk_w [T, k] fp32 in,
 *   optional; out [T, d] bf16 out.
 * A slot whose dest_row lies outside [0, T*k) is left out of its token's
 * sum (no memory outside y is read).
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_combine(const void* y, const int32_t* dest_row, const float* topk_w,
                         int64_t T, int32_t k, int32_t d, void* out, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 4 for training — the grouped gate/up GEMM of moe_grouped_swiglu
 * that also keeps the gate and up pre-activations G = x_perm Wg[e] and
 * U = x_perm Wu[e] (bf16), which the backward reads:
 *   h  [P, f] bf16 out, Silu(G)*U as moe_grouped_swiglu writes it;
 *   gu [P, 2f] bf16 out, interleaved like the packed gate/up weights: for
 *      gate/up tile t, gu[r, 128t + i] = G[r, 64t + i] and
 *      gu[r, 128t + 64 + i] = U[r, 64t + i], 0 <= i < 64.
 * Other arguments and errors as moe_grouped_swiglu; workspace
 * moe_grouped_swiglu_workspace_bytes().
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_grouped_gate_up_save(const void* x_perm, const int32_t* offsets, int64_t P,
                                      int32_t E, int32_t d, int32_t f, const void* packed,
                                      void* h, void* gu, void* workspace, size_t workspace_bytes,
                                      moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 4 backward — the grouped SwiGLU expert MLP (Algorithm 1, stage 4)
 * differentiated, as four grouped GEMMs on the tensor cores.  For expert e
 * and its rows (G, U from moe_grouped_gate_up_save, H = Silu(G)*U, dY the
 * gradient of the expert outputs):
 *   dH = dY Wd[e]^T;  dG = dH U Silu'(G);  dU = dH Silu(G)
 *   dx_perm = dG Wg[e]^T + dU Wu[e]^T
 *   dw_down[e] = H^T dY;  dw_gate[e] = X^T dG;  dw_up[e] = X^T dU
 * with fp32 accumulation and bf16 results.
 *   x_perm, dy, dx_perm [P, d] bf16; h [P, f]; gu, dgu [P, 2f] (dgu is
 *   written: dG and dU interleaved like gu); packed from moe_pack_weights
 *   (the same weights as the forward); dw_gate, dw_up [E, d, f] and
 *   dw_down [E, f, d] bf16 out, in moe_pack_weights' input layout (every
 *   expert written, zero for an expert without rows).
 * Workspace moe_grouped_swiglu_workspace_bytes().  Errors as
 * moe_grouped_swiglu.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_grouped_swiglu_backward(const void* x_perm, const void* h, const void* gu,
                                         const void* dy, const int32_t* offsets, int64_t P,
                                         int32_t E, int32_t d, int32_t f, const void* packed,
                                         void* dgu, void* dx_perm, void* dw_gate, void* dw_up,
                                         void* dw_down, void* workspace, size_t workspace_bytes,
                                         moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 5 backward — output reduction, backward (Algorithm 1, stage 5,
 * backward function): for every routed pair (t, j) at row
 * r = dest_row[t*k + j],
 *   d_mlp_out[r, :] = bf16( topk_w[t, j] * dout[t, :] )
 *   d_topk_w[t, j]  = sum_h mlp_out[r, h] * dout[t, h]   (fp32)
 *   dout [T, d] bf16; mlp_out [T*k, d] bf16, the expert outputs BEFORE the
 *   gate (moe_grouped_swiglu with row_scale = NULL); dest_row [T*k];
 *   topk_w [T, k] fp32; d_mlp_out [T*k, d] bf16 out; d_topk_w [T, k] out.
 * A slot whose dest_row lies outside [0, T*k) writes no row gradient and
 * gets d_topk_w = 0.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_combine_backward(const void* dout, const void* mlp_out, const int32_t* dest_row,
                                  const float* topk_w, int64_t T, int32_t k, int32_t d,
                                  void* d_mlp_out, float* d_topk_w, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 1 backward — gradient of the router logits from the gradient of
 * the gates, with the top-k selection held fixed (Softmax and TopK of
 * Algorithm 1, stage 1, differentiated): gates w_j = exp(l_{e_j}) / Z with
 * Z summed over all E experts, or over the k selected when renormalize != 0,
 * so d_logits[t, e] = [e is slot j] w_j dw_j - q_e * sum_j w_j dw_j with
 * q_e = exp(l_e) / Z on the normalisation set (0 elsewhere).
 *   logits [T, E] fp32 (as given to moe_route_topk); topk_idx [T, k];
 *   d_topk_w [T, k] fp32; d_logits [T, E] fp32 out (every entry written).
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_route_backward(const float* logits, const int32_t* topk_idx, const float* d_topk_w,
                                int64_t T, int32_t E, int32_t k, int32_t renormalize,
                                float* d_logits, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * The whole layer forward (Algorithm 1, stages 1-5) on one stream, with no
 * host synchronisation: route + per-chunk counts, index pass, permute,
 * gate/up GEMM with SwiGLU, down GEMM (rows left ungated), combine weighted
 * by the TopK weights.  The layout's y therefore holds each routed row's
 * expert output before its gate; row_w still holds the gate of every row.
 *   x [T, d] bf16; logits [T, E] fp32; packed from moe_pack_weights;
 *   out [T, d] bf16 out; topk_idx_out [T, k] int32 and topk_w_out [T, k]
 *   fp32 out, optional (the workspace keeps its own copy).
 * Workspace: moe_forward_workspace_bytes(T, E, k, d, f); the intermediates
 * stay there after the call at the byte offsets moe_forward_layout gives.
 * Errors: as the stages.
 * ---------------------------------------------------------------------- */
typedef struct {
  size_t topk_idx, topk_w, counts, offsets, src_token, dest_row, row_w;
  size_t x_perm, h, y;
  size_t total;
} moe_forward_layout_t;

MOE_API size_t moe_forward_workspace_bytes(int64_t T, int32_t E, int32_t k, int32_t d, int32_t f);
MOE_API moe_status_t moe_forward_layout(int64_t T, int32_t E, int32_t k, int32_t d, int32_t f,
                                moe_forward_layout_t* layout);
MOE_API moe_status_t moe_forward(const void* x, const float* logits, const void* packed,
                         int64_t T, int32_t d, int32_t E, int32_t k, int32_t f,
                         int32_t renormalize, void* out,
                         int32_t* topk_idx_out, float* topk_w_out,
                         void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_forward starting from the tokens and the router weights: stage 1 is
 * the fused router (moe_router_topk, with the token counts of stage 2 kept
 * on the side), so the router logits never exist in memory.  Other
 * arguments, the workspace and the layout are those of moe_forward.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_forward_routed(const void* x, const void* router_packed, const void* packed,
                                int64_t T, int32_t d, int32_t E, int32_t k, int32_t f,
                                int32_t renormalize, void* out,
                                int32_t* topk_idx_out, float* topk_w_out,
                                void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * The whole layer backward: the gradients of moe_forward's output with
 * respect to x, the router logits and the three expert weight tensors, for
 * an output gradient dout, the top-k selection held fixed.  The forward is
 * recomputed first (full activation recomputation: route, index, permute,
 * gate/up GEMM keeping G and U), then the output reduction backward
 * (Algorithm 1, stage 5), the gate gradient to the logits, the four
 * backward GEMMs of moe_grouped_swiglu_backward, and the un-permute of the
 * row gradients (each token sums its k rows).  Stage 5's gate gradient
 * <mlp_out[r], dout[t]> is formed as <H[r], dout[t] Wd^T> -- the same
 * product summed in the other order -- from the dgrad down GEMM, which then
 * takes the ungated rows of dout and applies the gates to its accumulator,
 * so the down projection is not recomputed (the down weight gradient H^T dY
 * is taken as (gated H)^T (ungated rows)); where that GEMM does not run on
 * SM pairs (f not a multiple of 256) the down GEMM is recomputed with
 * ungated rows and the gate gradient read from them.
 *   x [T, d] bf16; logits [T, E] fp32; packed from moe_pack_weights;
 *   dout [T, d] bf16; dx [T, d] bf16 out; d_logits [T, E] fp32 out;
 *   dw_gate, dw_up [E, d, f], dw_down [E, f, d] bf16 out.
 * Workspace moe_backward_workspace_bytes(T, E, k, d, f).  Errors as the
 * forward.  moe_backward_timed records events[i] (MOE_BACKWARD_STAGES + 1
 * caller-created cudaEvent_t) at the boundaries
 *   0 route+index+permute 1 gate/up 2 the output gradient on the expert
 *   rows (or the recomputed down GEMM, the output-reduction backward and
 *   the logit backward) 3 dgrad down 4 dgrad gate/up 5 gate gradient and
 *   logit backward (empty when done at 2) 6 wgrad down 7 wgrad gate/up 8
 *   un-permute 9; a NULL entry records nothing at its boundary, the array
 *   itself must not be NULL.
 * ---------------------------------------------------------------------- */
#define MOE_BACKWARD_STAGES 9
MOE_API size_t moe_backward_workspace_bytes(int64_t T, int32_t E, int32_t k, int32_t d, int32_t f);
MOE_API moe_status_t moe_backward(const void* x, const float* logits, const void* packed, const void* dout,
                          int64_t T, int32_t d, int32_t E, int32_t k, int32_t f, int32_t renormalize,
                          void* dx, float* d_logits, void* dw_gate, void* dw_up, void* dw_down,
                          void* workspace, size_t workspace_bytes, moe_stream_t stream);
MOE_API moe_status_t moe_backward_timed(const void* x, const float* logits, const void* packed,
                                const void* dout, int64_t T, int32_t d, int32_t E, int32_t k,
                                int32_t f, int32_t renormalize, void* dx, float* d_logits,
                                void* dw_gate, void* dw_up, void* dw_down, void* workspace,
                                size_t workspace_bytes, moe_stream_t stream, void* const* events);

/* ------------------------------------------------------------------------
 * moe_forward without the permuted copy of the tokens: the gate/up GEMM
 * fetches each A row x[src_token[r]] itself (four warps of 16-byte
 * asynchronous copies into the swizzled A stage) — the SonicMoE kernel's way
 * of running the expert GEMMs on the token-dispatch layout ("Training a
 * 1T-Params MoE on EU public infrastructure", SonicMoE).  Same arguments, results, workspace and
 * layout as moe_forward, except that the layout's x_perm region is left
 * unwritten.  moe_forward_gathered_timed records events as
 * moe_forward_timed does (the permute stage is empty).
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_forward_gathered(const void* x, const float* logits, const void* packed,
                                  int64_t T, int32_t d, int32_t E, int32_t k, int32_t f,
                                  int32_t renormalize, void* out,
                                  int32_t* topk_idx_out, float* topk_w_out,
                                  void* workspace, size_t workspace_bytes, moe_stream_t stream);
MOE_API moe_status_t moe_forward_gathered_timed(const void* x, const float* logits, const void* packed,
                                        int64_t T, int32_t d, int32_t E, int32_t k, int32_t f,
                                        int32_t renormalize, void* out, void* workspace,
                                        size_t workspace_bytes, moe_stream_t stream,
                                        void* const* events);

/* ------------------------------------------------------------------------
 * moe_forward with stage timing: identical work, plus cudaEventRecord of
 * events[i] (caller-created cudaEvent_t handles, MOE_FORWARD_STAGES + 1 of
 * them) on `stream` at the stage boundaries
 *   0 start | route | 1 | index | 2 | permute | 3 | gate/up GEMM |
 *   4 | down GEMM | 5 | combine | 6
 * so that cudaEventElapsedTime(events[i], events[i+1]) is the time of one
 * stage's kernel (stage 0 also holds the workspace clear).  A NULL entry
 * records nothing at that boundary (each recorded event separates two
 * kernels and costs a step some microseconds, so a caller timing one stage
 * passes only its two boundaries).  events itself must not be NULL.
 * ---------------------------------------------------------------------- */
#define MOE_FORWARD_STAGES 6
MOE_API moe_status_t moe_forward_timed(const void* x, const float* logits, const void* packed,
                               int64_t T, int32_t d, int32_t E, int32_t k, int32_t f,
                               int32_t renormalize, void* out,
                               void* workspace, size_t workspace_bytes, moe_stream_t stream,
                               void* const* events);

/* ------------------------------------------------------------------------
 * moe_forward from HOST buffers: copies x_host [T, d] bf16 and logits_host
 * [T, E] fp32 into device staging buffers, runs moe_forward, copies the
 * result into out_host [T, d] bf16, and waits for the stream.  Host buffers
 * should be page-locked for the copies to run at full speed.  The staging
 * buffers (x_dev, logits_dev, out_dev) are caller-owned device memory.
 * Errors: as moe_forward, plus MOE_ERR_CUDA for a failed copy.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_forward_host(const void* x_host, const float* logits_host, void* out_host,
                              void* x_dev, float* logits_dev, void* out_dev,
                              const void* packed, int64_t T, int32_t d, int32_t E, int32_t k,
                              int32_t f, int32_t renormalize,
                              void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_forward over a sequence of batches in HOST memory with the copies
 * overlapped with compute: batch b+1's inputs are copied in on copy_in and
 * batch b-1's output is copied out on copy_out while batch b runs on
 * `stream`, through two device staging slots.
 *   x_host[b] [T, d] bf16, logits_host[b] [T, E] fp32, out_host[b] [T, d]
 *   bf16: host pointers of batch b, 0 <= b < n_batches (pinned for full
 *   copy speed; a pointer may repeat);
 *   x_dev[2], logits_dev[2], out_dev[2]: the two device slots, each sized
 *   for one batch; workspace as moe_forward (shared by the batches, which
 *   run in order on `stream`).
 * stream, copy_in and copy_out must be three different streams.  Returns
 * once every copy has completed.  Errors: as moe_forward, and
 * MOE_ERR_INVALID_ARG for NULL arrays or pointers.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_forward_host_stream(const void* const* x_host, const float* const* logits_host,
                                     void* const* out_host, int32_t n_batches,
                                     void* const* x_dev, float* const* logits_dev,
                                     void* const* out_dev, const void* packed, int64_t T,
                                     int32_t d, int32_t E, int32_t k, int32_t f,
                                     int32_t renormalize, void* workspace,
                                     size_t workspace_bytes, moe_stream_t stream,
                                     moe_stream_t copy_in, moe_stream_t copy_out);

/* ------------------------------------------------------------------------
 * Check of the failure path every kernel shares: one block waits, with the
 * same bounded helpers the kernels use, on an mbarrier phase that never
 * completes, gives up after limit_ns (1 .. 2e9 ns, the kernels' own bound
 * being 2 s) and writes MOE_ERR_TIMEOUT into the workspace status word
 * (read it with moe_read_device_status); the context stays usable.
 * Workspace: 256 bytes, 256-byte aligned.  Errors: MOE_ERR_INVALID_ARG,
 * MOE_ERR_WORKSPACE, MOE_ERR_NO_DEVICE, MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int64_t limit_ns,
                                       moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Reads the device status word at the start of a workspace used by
 * moe_dispatch_scan, moe_grouped_swiglu or moe_forward, after waiting for
 * `stream`.  *status receives MOE_OK or the first device error.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_read_device_status(const void* workspace, moe_stream_t stream,
                                    int32_t* status);

/* ------------------------------------------------------------------------
 * The same read with the device status as the return value: waits for
 * `stream` and returns MOE_OK or the first error a kernel recorded in the
 * workspace (MOE_ERR_TIMEOUT, MOE_ERR_BAD_INDEX).  When the read itself
 * fails it returns MOE_ERR_INVALID_ARG (NULL workspace) or MOE_ERR_CUDA,
 * and moe_last_error says which.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_get_device_status(const void* workspace, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * The activation functions of the expert-GEMM epilogues ("Scalable
 * Pretraining of Large MoE LMs on Aurora Super Computer", §3.1, Algorithm 1,
 * stage 4: Silu(gate) * up, and its derivative through sigmoid), applied
 * elementwise with the very device functions the epilogues use, so that
 * their error can be measured: silu[i] = Silu(z[i]) = z[i] * sigmoid(z[i]),
 * sigmoid[i] = sigmoid(z[i]), fp32.  z, silu, sigmoid: device pointers to n
 * floats (no overlap between the inputs and the outputs); n >= 0.  Errors:
 * MOE_ERR_INVALID_ARG (n < 0, or NULL with n > 0), MOE_ERR_NO_DEVICE,
 * MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
MOE_API moe_status_t moe_selftest_activation(const float* z, int64_t n, float* silu, float* sigmoid,
                                             moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Measurement tools for the expert GEMMs' tile scheduling ("Training a
 * 1T-Params MoE on EU public infrastructure", *Dynamic tile scheduling in
 * SonicMoE*: tiles handed out at run time keep throughput when part of the
 * GPU is busy with other work; the page measures it against a dummy kernel
 * occupying 40 SMs).
 *
 * moe_set_tile_schedule: the tile schedule of the paired-SM expert GEMMs
 * launched afterwards by this process: MOE_TILE_SCHEDULE_DYNAMIC (the
 * default: every SM pair takes its next tile from a shared atomic counter)
 * or MOE_TILE_SCHEDULE_STATIC (pair i takes tiles i, i + pairs, i + 2 pairs,
 * ... whatever the others do).  Results are identical under both; only the
 * order in which tiles run differs.  Not thread-safe against concurrent
 * launches.  Errors: MOE_ERR_INVALID_ARG (another mode).
 *
 * moe_occupy_sms: a kernel of n_sms blocks on `stream` (0 <= n_sms <= the
 * device's SM count), each holding one SM (it takes most of the SM's shared
 * memory, so no expert-GEMM block fits beside it) and returning after
 * duration_ns (0 .. 10^10 ns); kernels on other streams run on the other
 * SMs meanwhile.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_NO_DEVICE,
 * MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
#define MOE_TILE_SCHEDULE_DYNAMIC 0
#define MOE_TILE_SCHEDULE_STATIC 1
MOE_API moe_status_t moe_set_tile_schedule(int32_t mode);
MOE_API moe_status_t moe_occupy_sms(int32_t n_sms, int64_t duration_ns, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
