// C ABI of the MoE-layer forward: argument checks, workspace layout and the
// order of launches.  Every entry point validates on the host before it
// touches CUDA, so argument errors never reach the GPU.
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <string>

#include "moe_gb300.h"
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

thread_local std::string g_last_error;

moe_status_t fail(moe_status_t s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

moe_status_t cuda_fail(cudaError_t e, const char* where) {
  g_last_error = std::string(where) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return MOE_ERR_CUDA;
}

#define MOE_CUDA(call, where)                   \
  do {                                          \
    cudaError_t err_ = (call);                  \
    if (err_ != cudaSuccess) return cuda_fail(err_, where); \
  } while (0)

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int32_t kRouterMaxExperts = 512;  // the fused router's accumulator fits TMEM's 512 columns

moe_status_t check_row(int32_t d, const char* name) {
  if (d < 8 || d > 65536 || d % 8 != 0)
    return fail(MOE_ERR_UNSUPPORTED, std::string(name) + " must be a multiple of 8 in [8, 65536]");
  return MOE_OK;
}

moe_status_t check_gemm_dims(int32_t d, int32_t f) {
  if (d < 64 || d > 65536 || d % 64 != 0) return fail(MOE_ERR_UNSUPPORTED, "d must be a multiple of 64 in [64, 65536]");
  if (f < 64 || f > 65536 || f % 64 != 0) return fail(MOE_ERR_UNSUPPORTED, "f must be a multiple of 64 in [64, 65536]");
  return MOE_OK;
}

// Upper bound on the flat tile index of the grouped GEMMs must fit int32.
moe_status_t check_tile_space(int64_t P, int32_t E, int32_t d, int32_t f) {
  const int64_t mt = P / 128 + E;
  const int64_t nt = std::max<int64_t>(2 * static_cast<int64_t>(f) / 128, static_cast<int64_t>(d) / 64);
  if (mt * nt >= (int64_t(1) << 31)) return fail(MOE_ERR_UNSUPPORTED, "problem too large for the tile index");
  return MOE_OK;
}

// The FP8-weight layout and GEMMs: d and f multiples of 128 (whole scale
// blocks per stored row, 128-row code tiles), d a multiple of 256 (the
// paired down GEMM), and every code row addressable by the tensor maps.
moe_status_t check_fp8_pack_dims(int32_t E, int32_t d, int32_t f) {
  if (E < 1 || E > MOE_MAX_EXPERTS) return fail(MOE_ERR_UNSUPPORTED, "E must be in [1, 1024]");
  if (d < 128 || d > 65536 || d % 128 != 0) return fail(MOE_ERR_UNSUPPORTED, "FP8 weights need d a multiple of 128");
  if (f < 128 || f > 65536 || f % 128 != 0) return fail(MOE_ERR_UNSUPPORTED, "FP8 weights need f a multiple of 128");
  if (static_cast<int64_t>(E) * 2 * f * (d / 64) >= (int64_t(1) << 31) ||
      static_cast<int64_t>(E) * d * (f / 64) >= (int64_t(1) << 31))
    return fail(MOE_ERR_UNSUPPORTED, "FP8 weights too large for the code tensor maps");
  return MOE_OK;
}

moe_status_t check_fp8_forward_dims(int32_t E, int32_t d, int32_t f) {
  moe_status_t s = check_fp8_pack_dims(E, d, f);
  if (s != MOE_OK) return s;
  if (d % 256 != 0) return fail(MOE_ERR_UNSUPPORTED, "the FP8-weight forward needs d a multiple of 256");
  return MOE_OK;
}

moe_status_t device_info(DeviceInfo* info) {
  cudaError_t e = current_device_info(info);
  if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver)
    return fail(MOE_ERR_NO_DEVICE, "no CUDA device available");
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  if (info->cc_major != 10 || info->cc_minor != 3)
    return fail(MOE_ERR_NO_DEVICE, "the library is built for sm_103a (GB300); device has compute capability " +
                                       std::to_string(info->cc_major) + "." + std::to_string(info->cc_minor));
  return MOE_OK;
}

// ---- moe_forward workspace layout
struct ForwardLayout {
  size_t header, hist, counts, offsets;
  size_t topk_idx, topk_w, src_token, dest_row, row_w, x_perm, h, y, total;
  size_t clear_bytes;
};

ForwardLayout forward_layout(int64_t T, int32_t E, int32_t k, int32_t d, int32_t f) {
  const int64_t P = T * k;
  ForwardLayout L{};
  size_t o = 0;
  L.header = o;
  o = sizeof(WsHeader);
  L.hist = o;                   // the per-chunk count table, filled by atomic adds of the route kernel
  o += dispatch_hist_bytes(P, E);
  L.clear_bytes = o;            // the header and the table start at zero
  L.counts = o;
  o += align_up(static_cast<size_t>(E) * 4);
  L.offsets = o;
  o += align_up(static_cast<size_t>(E + 1) * 4);
  L.topk_idx = o;
  o += align_up(static_cast<size_t>(P) * 4);
  L.topk_w = o;
  o += align_up(static_cast<size_t>(P) * 4);
  L.src_token = o;
  o += align_up(static_cast<size_t>(P) * 4);
  L.dest_row = o;
  o += align_up(static_cast<size_t>(P) * 4);
  L.row_w = o;
  o += align_up(static_cast<size_t>(P) * 4);
  L.x_perm = o;
  o += align_up(static_cast<size_t>(P) * d * 2);
  L.h = o;
  o += align_up(static_cast<size_t>(P) * f * 2);
  L.y = o;
  o += align_up(static_cast<size_t>(P) * d * 2);
  L.total = o;
  return L;
}

// ---- moe_backward workspace layout (the forward's buffers, then the
// backward's).  y holds the recomputed expert outputs where the down
// projection is recomputed, and is reused for dx_perm; dy holds the gated
// output-gradient rows, or, without the recomputation, the ungated ones.
// dh holds the down projection's input gradient before the gates (only
// used without the recomputation).
struct BackwardLayout {
  ForwardLayout F;
  size_t gu, dy, dgu, d_topk_w, dh, total;
};

BackwardLayout backward_layout(int64_t T, int32_t E, int32_t k, int32_t d, int32_t f) {
  const int64_t P = T * k;
  BackwardLayout L{};
  L.F = forward_layout(T, E, k, d, f);
  size_t o = L.F.total;
  L.gu = o;
  o += align_up(static_cast<size_t>(P) * 2 * f * 2);
  L.dy = o;
  o += align_up(static_cast<size_t>(P) * d * 2);
  L.dgu = o;
  o += align_up(static_cast<size_t>(P) * 2 * f * 2);
  L.d_topk_w = o;
  o += align_up(static_cast<size_t>(P) * 4);
  L.dh = o;
  o += align_up(static_cast<size_t>(P) * f * 2);
  L.total = o;
  return L;
}

}  // namespace

void set_last_error(const std::string& msg) { g_last_error = msg; }

moe_status_t check_routing(int64_t T, int32_t E, int32_t k) {
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T must be >= 0");
  if (E < 1 || E > MOE_MAX_EXPERTS)
    return fail(MOE_ERR_UNSUPPORTED, "E must be in [1, " + std::to_string(MOE_MAX_EXPERTS) + "]");
  if (k < 1 || k > E || k > MOE_MAX_TOPK)
    return fail(MOE_ERR_UNSUPPORTED, "k must be in [1, min(E, " + std::to_string(MOE_MAX_TOPK) + ")]");
  if (T * static_cast<int64_t>(k) >= (int64_t(1) << 31)) return fail(MOE_ERR_UNSUPPORTED, "T*k must be < 2^31");
  return MOE_OK;
}

cudaError_t current_device_info(DeviceInfo* info) {
  static DeviceInfo cache[64];
  static bool have[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && have[dev]) {
    *info = cache[dev];
    return cudaSuccess;
  }
  DeviceInfo d{};
  d.device = dev;
  e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) {
    cache[dev] = d;
    have[dev] = true;
  }
  *info = d;
  return cudaSuccess;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return MOE_GB300_ABI_VERSION; }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
    case MOE_ERR_BAD_INDEX: return "expert index out of range";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_NO_DEVICE: return "no supported CUDA device";
  }
  return "unknown status";
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

moe_status_t moe_route_topk(const float* logits, int64_t T, int32_t E, int32_t k, int32_t renormalize,
                            int32_t* topk_idx, float* topk_w, moe_stream_t stream) {
  moe_status_t s = check_routing(T, E, k);
  if (s != MOE_OK) return s;
  if (T > 0 && (!logits || !topk_idx || !topk_w)) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (T == 0) return MOE_OK;
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  MOE_CUDA(launch_route_topk(logits, T, E, k, 1, renormalize, topk_idx, topk_w, nullptr, dev.num_sms,
                             static_cast<cudaStream_t>(stream)),
           "route_topk launch");
  return MOE_OK;
}

moe_status_t moe_route_topk_grouped(const float* logits, int64_t T, int32_t E, int32_t k, int32_t n_groups,
                                    int32_t renormalize, int32_t* topk_idx, float* topk_w, moe_stream_t stream) {
  moe_status_t s = check_routing(T, E, k);
  if (s != MOE_OK) return s;
  if (n_groups < 1 || E % n_groups != 0 || k % n_groups != 0)
    return fail(MOE_ERR_UNSUPPORTED, "n_groups must be >= 1 and divide both E and k");
  if (T > 0 && (!logits || !topk_idx || !topk_w)) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (T == 0) return MOE_OK;
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  MOE_CUDA(launch_route_topk(logits, T, E, k, n_groups, renormalize, topk_idx, topk_w, nullptr, dev.num_sms,
                             static_cast<cudaStream_t>(stream)),
           "route_topk_grouped launch");
  return MOE_OK;
}

size_t moe_router_packed_bytes(int32_t d, int32_t E) {
  if (d < 1 || E < 1) return 0;
  return static_cast<size_t>(d) * router_e_pad(E) * 2;
}

moe_status_t moe_pack_router_weights(const void* w_router, int32_t d, int32_t E, void* packed, moe_stream_t stream) {
  if (E < 1 || E > kRouterMaxExperts) return fail(MOE_ERR_UNSUPPORTED, "the fused router takes 1 <= E <= 512");
  if (d < 64 || d > 65536 || d % 64 != 0) return fail(MOE_ERR_UNSUPPORTED, "d must be a multiple of 64 in [64, 65536]");
  if (!w_router || !packed) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  DeviceInfo dev;
  moe_status_t s = device_info(&dev);
  if (s != MOE_OK) return s;
  MOE_CUDA(launch_pack_router(w_router, d, E, packed, static_cast<cudaStream_t>(stream)), "router pack launch");
  return MOE_OK;
}

moe_status_t moe_router_topk(const void* x, const void* router_packed, int64_t T, int32_t d, int32_t E, int32_t k,
                             int32_t renormalize, int32_t* topk_idx, float* topk_w, void* workspace,
                             size_t workspace_bytes, moe_stream_t stream) {
  moe_status_t s = check_routing(T, E, k);
  if (s != MOE_OK) return s;
  if (E > kRouterMaxExperts) return fail(MOE_ERR_UNSUPPORTED, "the fused router takes E <= 512");
  if (d < 64 || d > 65536 || d % 64 != 0) return fail(MOE_ERR_UNSUPPORTED, "d must be a multiple of 64 in [64, 65536]");
  if (!router_packed) return fail(MOE_ERR_INVALID_ARG, "NULL router weights");
  if (T > 0 && (!x || !topk_idx || !topk_w)) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(x, 16) || !aligned(router_packed, 16)) return fail(MOE_ERR_INVALID_ARG, "x and weights must be 16-byte aligned");
  if (!workspace || workspace_bytes < sizeof(WsHeader) || !aligned(workspace, kAlign))
    return fail(MOE_ERR_WORKSPACE, "router workspace needs 256 bytes, 256-byte aligned");
  if (T == 0) return MOE_OK;
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_CUDA(cudaMemsetAsync(workspace, 0, sizeof(WsHeader), st), "workspace clear");
  MOE_CUDA(launch_router_topk(x, router_packed, T, d, E, k, renormalize, topk_idx, topk_w, nullptr,
                              &static_cast<WsHeader*>(workspace)->status, st),
           "router launch");
  return MOE_OK;
}

size_t moe_dispatch_workspace_bytes(int64_t T, int32_t E, int32_t k) {
  if (T < 0 || E < 1 || k < 1) return 0;
  return sizeof(WsHeader) + dispatch_hist_bytes(T * k, E);
}

moe_status_t moe_dispatch_scan(const int32_t* topk_idx, const float* topk_w, int64_t T, int32_t E, int32_t k,
                               int32_t* counts, int32_t* offsets, int32_t* src_token, int32_t* dest_row,
                               float* row_w, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  moe_status_t s = check_routing(T, E, k);
  if (s != MOE_OK) return s;
  if (!counts || !offsets) return fail(MOE_ERR_INVALID_ARG, "NULL counts/offsets");
  if (T > 0 && (!topk_idx || !src_token || !dest_row)) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (row_w && !topk_w) return fail(MOE_ERR_INVALID_ARG, "row_w needs topk_w");
  const size_t need = moe_dispatch_workspace_bytes(T, E, k);
  if (!workspace || workspace_bytes < need || !aligned(workspace, kAlign))
    return fail(MOE_ERR_WORKSPACE, "dispatch workspace needs " + std::to_string(need) + " bytes, 256-byte aligned");
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t P = T * k;
  MOE_CUDA(cudaMemsetAsync(workspace, 0, sizeof(WsHeader), st), "workspace clear");
  if (P == 0) {
    MOE_CUDA(cudaMemsetAsync(counts, 0, static_cast<size_t>(E) * 4, st), "counts clear");
    MOE_CUDA(cudaMemsetAsync(offsets, 0, static_cast<size_t>(E + 1) * 4, st), "offsets clear");
    return MOE_OK;
  }
  auto* hdr = static_cast<WsHeader*>(workspace);
  auto* hist = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + sizeof(WsHeader));
  MOE_CUDA(launch_chunk_histogram(topk_idx, P, E, hist, &hdr->status, st), "histogram launch");
  MOE_CUDA(launch_index(topk_idx, topk_w, P, E, k, hist, counts, offsets, src_token, dest_row, row_w, &hdr->status,
                        st),
           "index launch");
  return MOE_OK;
}

moe_status_t moe_permute(const void* x, int64_t T, int32_t d, const int32_t* dest_row, int32_t k, void* x_perm,
                         moe_stream_t stream) {
  if (T < 0 || k < 1 || k > MOE_MAX_TOPK) return fail(MOE_ERR_INVALID_ARG, "bad T or k");
  if (T * static_cast<int64_t>(k) >= (int64_t(1) << 31)) return fail(MOE_ERR_UNSUPPORTED, "T*k must be < 2^31");
  moe_status_t s = check_row(d, "d");
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!x || !dest_row || !x_perm) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(x, 16) || !aligned(x_perm, 16)) return fail(MOE_ERR_INVALID_ARG, "x and x_perm must be 16-byte aligned");
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  MOE_CUDA(launch_permute(x, T, d, dest_row, k, x_perm, nullptr, dev.num_sms, static_cast<cudaStream_t>(stream)),
           "permute launch");
  return MOE_OK;
}

size_t moe_packed_weight_bytes(int32_t E, int32_t d, int32_t f) {
  if (E < 1 || d < 1 || f < 1) return 0;
  return static_cast<size_t>(3) * E * static_cast<size_t>(d) * f * 2;
}

moe_status_t moe_pack_weights(const void* w_gate, const void* w_up, const void* w_down, int32_t E, int32_t d,
                              int32_t f, void* packed, moe_stream_t stream) {
  if (E < 1 || E > MOE_MAX_EXPERTS) return fail(MOE_ERR_UNSUPPORTED, "E must be in [1, 1024]");
  moe_status_t s = check_gemm_dims(d, f);
  if (s != MOE_OK) return s;
  if (!w_gate || !w_up || !w_down || !packed) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  MOE_CUDA(launch_pack_weights(w_gate, w_up, w_down, E, d, f, packed, static_cast<cudaStream_t>(stream)),
           "pack launch");
  return MOE_OK;
}

moe_status_t moe_quantize_fp8_blockwise(const void* w, int64_t n, uint8_t* codes, float* scales, moe_stream_t stream) {
  if (n < 0 || n % 128 != 0) return fail(MOE_ERR_INVALID_ARG, "n must be a non-negative multiple of 128");
  if (n > 0 && (!w || !codes || !scales)) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(w, 8) || !aligned(codes, 4)) return fail(MOE_ERR_INVALID_ARG, "w must be 8-byte and codes 4-byte aligned");
  if (n == 0) return MOE_OK;
  DeviceInfo dev;
  moe_status_t s = device_info(&dev);
  if (s != MOE_OK) return s;
  MOE_CUDA(launch_quantize_fp8(w, n, codes, scales, dev.num_sms, static_cast<cudaStream_t>(stream)),
           "fp8 quantize launch");
  return MOE_OK;
}

moe_status_t moe_dequantize_fp8_blockwise(const uint8_t* codes, const float* scales, int64_t n, void* w_out,
                                          moe_stream_t stream) {
  if (n < 0 || n % 128 != 0) return fail(MOE_ERR_INVALID_ARG, "n must be a non-negative multiple of 128");
  if (n > 0 && (!w_out || !codes || !scales)) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(w_out, 8) || !aligned(codes, 4)) return fail(MOE_ERR_INVALID_ARG, "w_out must be 8-byte and codes 4-byte aligned");
  if (n == 0) return MOE_OK;
  DeviceInfo dev;
  moe_status_t s = device_info(&dev);
  if (s != MOE_OK) return s;
  MOE_CUDA(launch_dequantize_fp8(codes, scales, n, w_out, dev.num_sms, static_cast<cudaStream_t>(stream)),
           "fp8 dequantize launch");
  return MOE_OK;
}

size_t moe_grouped_swiglu_workspace_bytes(void) { return sizeof(WsHeader); }

moe_status_t moe_grouped_swiglu(const void* x_perm, const int32_t* offsets, int64_t P, int32_t E, int32_t d,
                                int32_t f, const void* packed, const float* row_scale, void* h, void* y,
                                void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (P < 0 || P >= (int64_t(1) << 31)) return fail(MOE_ERR_UNSUPPORTED, "P must be in [0, 2^31)");
  if (E < 1 || E > MOE_MAX_EXPERTS) return fail(MOE_ERR_UNSUPPORTED, "E must be in [1, 1024]");
  moe_status_t s = check_gemm_dims(d, f);
  if (s != MOE_OK) return s;
  if ((s = check_tile_space(P, E, d, f)) != MOE_OK) return s;
  if (!offsets || !packed) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (P > 0 && (!x_perm || !h || !y)) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!workspace || workspace_bytes < sizeof(WsHeader) || !aligned(workspace, kAlign))
    return fail(MOE_ERR_WORKSPACE, "grouped GEMM workspace needs 256 bytes, 256-byte aligned");
  if (!aligned(x_perm, 16) || !aligned(h, 16) || !aligned(y, 16) || !aligned(packed, 16))
    return fail(MOE_ERR_INVALID_ARG, "x_perm, h, y and packed must be 16-byte aligned");
  if (P == 0) return MOE_OK;
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto* hdr = static_cast<WsHeader*>(workspace);
  MOE_CUDA(cudaMemsetAsync(workspace, 0, sizeof(WsHeader), st), "workspace clear");
  const auto* wgu = static_cast<const __nv_bfloat16*>(packed);
  const auto* wdn = wgu + static_cast<int64_t>(E) * 2 * f * d;
  GroupedGemmProblem g1{x_perm, wgu, offsets, nullptr, h, P, E, d, 2 * f, f, &hdr->tile_counter[0], &hdr->status};
  MOE_CUDA(launch_grouped_gemm(g1, Epilogue::kSwiGLU, dev.num_sms, st), "gate/up GEMM launch");
  GroupedGemmProblem g2{h, wdn, offsets, row_scale, y, P, E, f, d, d, &hdr->tile_counter[1], &hdr->status};
  MOE_CUDA(launch_grouped_gemm(g2, Epilogue::kScale, dev.num_sms, st), "down GEMM launch");
  return MOE_OK;
}

moe_status_t moe_combine(const void* y, const int32_t* dest_row, const float* topk_w, int64_t T, int32_t k,
                         int32_t d, void* out, moe_stream_t stream) {
  if (T < 0 || k < 1 || k > MOE_MAX_TOPK) return fail(MOE_ERR_INVALID_ARG, "bad T or k");
  if (T * static_cast<int64_t>(k) >= (int64_t(1) << 31)) return fail(MOE_ERR_UNSUPPORTED, "T*k must be < 2^31");
  moe_status_t s = check_row(d, "d");
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!y || !dest_row || !out) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(y, 16) || !aligned(out, 16)) return fail(MOE_ERR_INVALID_ARG, "y and out must be 16-byte aligned");
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  MOE_CUDA(launch_combine(y, dest_row, topk_w, T, k, d, out, nullptr, dev.num_sms, static_cast<cudaStream_t>(stream)),
           "combine launch");
  return MOE_OK;
}

moe_status_t moe_combine_backward(const void* dout, const void* mlp_out, const int32_t* dest_row, const float* topk_w,
                                  int64_t T, int32_t k, int32_t d, void* d_mlp_out, float* d_topk_w,
                                  moe_stream_t stream) {
  if (T < 0 || k < 1 || k > MOE_MAX_TOPK) return fail(MOE_ERR_INVALID_ARG, "bad T or k");
  if (T * static_cast<int64_t>(k) >= (int64_t(1) << 31)) return fail(MOE_ERR_UNSUPPORTED, "T*k must be < 2^31");
  moe_status_t s = check_row(d, "d");
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!dout || !mlp_out || !dest_row || !topk_w || !d_mlp_out || !d_topk_w)
    return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(dout, 16) || !aligned(mlp_out, 16) || !aligned(d_mlp_out, 16))
    return fail(MOE_ERR_INVALID_ARG, "dout, mlp_out and d_mlp_out must be 16-byte aligned");
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  MOE_CUDA(launch_combine_backward(dout, mlp_out, dest_row, topk_w, T, k, d, d_mlp_out, d_topk_w, nullptr, dev.num_sms,
                                   static_cast<cudaStream_t>(stream)),
           "combine backward launch");
  return MOE_OK;
}

moe_status_t moe_route_backward(const float* logits, const int32_t* topk_idx, const float* d_topk_w, int64_t T,
                                int32_t E, int32_t k, int32_t renormalize, float* d_logits, moe_stream_t stream) {
  moe_status_t s = check_routing(T, E, k);
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_idx || !d_topk_w || !d_logits) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  MOE_CUDA(launch_route_backward(logits, topk_idx, d_topk_w, T, E, k, renormalize, d_logits, dev.num_sms,
                                 static_cast<cudaStream_t>(stream)),
           "route backward launch");
  return MOE_OK;
}

moe_status_t moe_grouped_gate_up_save(const void* x_perm, const int32_t* offsets, int64_t P, int32_t E, int32_t d,
                                      int32_t f, const void* packed, void* h, void* gu, void* workspace,
                                      size_t workspace_bytes, moe_stream_t stream) {
  if (P < 0 || P >= (int64_t(1) << 31)) return fail(MOE_ERR_UNSUPPORTED, "P must be in [0, 2^31)");
  if (E < 1 || E > MOE_MAX_EXPERTS) return fail(MOE_ERR_UNSUPPORTED, "E must be in [1, 1024]");
  moe_status_t s = check_gemm_dims(d, f);
  if (s != MOE_OK) return s;
  if ((s = check_tile_space(P, E, d, f)) != MOE_OK) return s;
  if (!offsets || !packed) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (P > 0 && (!x_perm || !h || !gu)) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!workspace || workspace_bytes < sizeof(WsHeader) || !aligned(workspace, kAlign))
    return fail(MOE_ERR_WORKSPACE, "grouped GEMM workspace needs 256 bytes, 256-byte aligned");
  if (!aligned(x_perm, 16) || !aligned(h, 16) || !aligned(gu, 16) || !aligned(packed, 16))
    return fail(MOE_ERR_INVALID_ARG, "x_perm, h, gu and packed must be 16-byte aligned");
  if (P == 0) return MOE_OK;
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto* hdr = static_cast<WsHeader*>(workspace);
  MOE_CUDA(cudaMemsetAsync(workspace, 0, sizeof(WsHeader), st), "workspace clear");
  BackwardGemmArgs a{};
  a.P = P;
  a.E = E;
  a.d = d;
  a.f = f;
  a.offsets = offsets;
  a.w_gate_up = packed;
  a.x_perm = x_perm;
  a.h = h;
  a.gu = gu;
  a.counters = hdr->tile_counter;
  a.status = &hdr->status;
  MOE_CUDA(launch_gate_up_save(a, dev.num_sms, st), "gate/up GEMM launch");
  return MOE_OK;
}

moe_status_t moe_grouped_swiglu_backward(const void* x_perm, const void* h, const void* gu, const void* dy,
                                         const int32_t* offsets, int64_t P, int32_t E, int32_t d, int32_t f,
                                         const void* packed, void* dgu, void* dx_perm, void* dw_gate, void* dw_up,
                                         void* dw_down, void* workspace, size_t workspace_bytes,
                                         moe_stream_t stream) {
  if (P < 0 || P >= (int64_t(1) << 31)) return fail(MOE_ERR_UNSUPPORTED, "P must be in [0, 2^31)");
  if (E < 1 || E > MOE_MAX_EXPERTS) return fail(MOE_ERR_UNSUPPORTED, "E must be in [1, 1024]");
  moe_status_t s = check_gemm_dims(d, f);
  if (s != MOE_OK) return s;
  if ((s = check_tile_space(P, E, d, f)) != MOE_OK) return s;
  if (static_cast<int64_t>(E) * ((std::max(d, f) + 127) / 128) * (2 * static_cast<int64_t>(f) / 64 + d / 64) >=
      (int64_t(1) << 31))
    return fail(MOE_ERR_UNSUPPORTED, "problem too large for the tile index");
  if (!offsets || !packed || !dw_gate || !dw_up || !dw_down) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (P > 0 && (!x_perm || !h || !gu || !dy || !dgu || !dx_perm)) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!workspace || workspace_bytes < sizeof(WsHeader) || !aligned(workspace, kAlign))
    return fail(MOE_ERR_WORKSPACE, "grouped GEMM workspace needs 256 bytes, 256-byte aligned");
  const void* al[] = {x_perm, h, gu, dy, dgu, dx_perm, dw_gate, dw_up, dw_down, packed};
  for (const void* q : al)
    if (!aligned(q, 16)) return fail(MOE_ERR_INVALID_ARG, "every matrix must be 16-byte aligned");
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto* hdr = static_cast<WsHeader*>(workspace);
  MOE_CUDA(cudaMemsetAsync(workspace, 0, sizeof(WsHeader), st), "workspace clear");
  BackwardGemmArgs a{};
  a.P = P;
  a.E = E;
  a.d = d;
  a.f = f;
  a.offsets = offsets;
  a.w_gate_up = packed;
  a.w_down = static_cast<const __nv_bfloat16*>(packed) + static_cast<int64_t>(E) * 2 * f * d;
  a.x_perm = x_perm;
  a.dy = dy;
  a.h = const_cast<void*>(h);
  a.gu = const_cast<void*>(gu);
  a.dgu = dgu;
  a.dx_perm = dx_perm;
  a.dw_gate = dw_gate;
  a.dw_up = dw_up;
  a.dw_down = dw_down;
  a.counters = hdr->tile_counter;
  a.status = &hdr->status;
  MOE_CUDA(launch_swiglu_backward_gemms(a, dev.num_sms, st, nullptr), "backward GEMM launch");
  return MOE_OK;
}

size_t moe_forward_workspace_bytes(int64_t T, int32_t E, int32_t k, int32_t d, int32_t f) {
  if (T < 0 || E < 1 || k < 1 || d < 1 || f < 1) return 0;
  return forward_layout(T, E, k, d, f).total;
}

moe_status_t moe_forward_layout(int64_t T, int32_t E, int32_t k, int32_t d, int32_t f,
                                moe_forward_layout_t* layout) {
  if (!layout) return fail(MOE_ERR_INVALID_ARG, "NULL layout");
  moe_status_t s = check_routing(T, E, k);
  if (s != MOE_OK) return s;
  if ((s = check_gemm_dims(d, f)) != MOE_OK) return s;
  const ForwardLayout L = forward_layout(T, E, k, d, f);
  layout->topk_idx = L.topk_idx;
  layout->topk_w = L.topk_w;
  layout->counts = L.counts;
  layout->offsets = L.offsets;
  layout->src_token = L.src_token;
  layout->dest_row = L.dest_row;
  layout->row_w = L.row_w;
  layout->x_perm = L.x_perm;
  layout->h = L.h;
  layout->y = L.y;
  layout->total = L.total;
  return MOE_OK;
}

}  // extern "C"

namespace {

// Stage 1 reads `logits` when router_packed is null, else computes the
// logits from x and the packed router weights inside the route kernel.
// With `gathered`, the gate/up GEMM reads its A rows from x through
// src_token (TMA gathers) and no permuted copy is made.
moe_status_t forward_impl(const void* x, const float* logits, const void* router_packed, const void* packed,
                          int64_t T, int32_t d, int32_t E, int32_t k, int32_t f, int32_t renormalize, void* out,
                          int32_t* topk_idx_out, float* topk_w_out, void* workspace, size_t workspace_bytes,
                          moe_stream_t stream, void* const* events, bool gathered = false, bool fp8 = false) {
  moe_status_t s = check_routing(T, E, k);
  if (s != MOE_OK) return s;
  if ((s = check_gemm_dims(d, f)) != MOE_OK) return s;
  const int64_t P = T * k;
  if ((s = check_tile_space(P, E, d, f)) != MOE_OK) return s;
  if (fp8 && (s = check_fp8_forward_dims(E, d, f)) != MOE_OK) return s;
  if (fp8 && !aligned(packed, kAlign)) return fail(MOE_ERR_INVALID_ARG, "FP8 packed weights must be 256-byte aligned");
  if (!packed) return fail(MOE_ERR_INVALID_ARG, "NULL packed weights");
  if (T > 0 && (!x || (!logits && !router_packed) || !out)) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (router_packed && E > kRouterMaxExperts) return fail(MOE_ERR_UNSUPPORTED, "the fused router takes E <= 512");
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(packed, 16))
    return fail(MOE_ERR_INVALID_ARG, "x, out and packed must be 16-byte aligned");
  const ForwardLayout L = forward_layout(T, E, k, d, f);
  if (!workspace || workspace_bytes < L.total || !aligned(workspace, kAlign))
    return fail(MOE_ERR_WORKSPACE, "forward workspace needs " + std::to_string(L.total) + " bytes, 256-byte aligned");
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  auto* hdr = reinterpret_cast<WsHeader*>(ws);
  auto* hist = reinterpret_cast<int32_t*>(ws + L.hist);
  auto* counts = reinterpret_cast<int32_t*>(ws + L.counts);
  auto* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  int32_t* topk_idx = topk_idx_out ? topk_idx_out : reinterpret_cast<int32_t*>(ws + L.topk_idx);
  float* topk_w = topk_w_out ? topk_w_out : reinterpret_cast<float*>(ws + L.topk_w);
  auto* src_token = reinterpret_cast<int32_t*>(ws + L.src_token);
  auto* dest_row = reinterpret_cast<int32_t*>(ws + L.dest_row);
  auto* row_w = reinterpret_cast<float*>(ws + L.row_w);
  void* x_perm = ws + L.x_perm;
  void* h = ws + L.h;
  void* y = ws + L.y;

  auto mark = [&](int i) -> cudaError_t {
    return events && events[i] ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) : cudaSuccess;
  };
  MOE_CUDA(mark(0), "event record");
  MOE_CUDA(cudaMemsetAsync(ws, 0, L.clear_bytes, st), "workspace clear");
  if (T == 0) {
    MOE_CUDA(cudaMemsetAsync(counts, 0, static_cast<size_t>(E) * 4, st), "counts clear");
    MOE_CUDA(cudaMemsetAsync(offsets, 0, static_cast<size_t>(E + 1) * 4, st), "offsets clear");
    for (int i = 1; i <= MOE_FORWARD_STAGES; ++i) MOE_CUDA(mark(i), "event record");
    return MOE_OK;
  }
  // stage 1 (+ the per-chunk token counts)
  if (router_packed) {
    MOE_CUDA(launch_router_topk(x, router_packed, T, d, E, k, renormalize, topk_idx, topk_w, hist, &hdr->status, st),
             "router launch");
  } else {
    MOE_CUDA(launch_route_topk(logits, T, E, k, 1, renormalize, topk_idx, topk_w, hist, dev.num_sms, st),
             "route launch");
  }
  MOE_CUDA(mark(1), "event record");
  // stages 2-3: counts, offsets, index maps and the gate of every row
  MOE_CUDA(launch_index(topk_idx, topk_w, P, E, k, hist, counts, offsets, src_token, dest_row, row_w, &hdr->status,
                        st),
           "index launch");
  MOE_CUDA(mark(2), "event record");
  // stage 4
  if (!gathered)
    MOE_CUDA(launch_permute(x, T, d, dest_row, k, x_perm, &hdr->status, dev.num_sms, st), "permute launch");
  MOE_CUDA(mark(3), "event record");
  const auto* wgu = static_cast<const __nv_bfloat16*>(packed);
  const auto* wdn = wgu + static_cast<int64_t>(E) * 2 * f * d;
  GroupedGemmProblem g1{x_perm, wgu, offsets, nullptr, h, P, E, d, 2 * f, f, &hdr->tile_counter[0], &hdr->status};
  // the down GEMM leaves its rows ungated: the gates enter in the output
  // reduction, where they cost no extra memory traffic
  GroupedGemmProblem g2{h, wdn, offsets, nullptr, y, P, E, f, d, d, &hdr->tile_counter[1], &hdr->status};
  if (fp8) {
    size_t off[4];
    fp8_packed_bytes(E, d, f, off);
    const auto* pk = static_cast<const uint8_t*>(packed);
    g1.b = pk + off[0];
    g1.fp8_scales = reinterpret_cast<const float*>(pk + off[2]);
    g2.b = pk + off[1];
    g2.fp8_scales = reinterpret_cast<const float*>(pk + off[3]);
  }
  if (gathered) {
    g1.a = x;
    g1.gather_rows = src_token;
    g1.a_rows = T;
  }
  MOE_CUDA(fp8 ? launch_grouped_gemm_2sm_fp8(g1, Epilogue::kSwiGLU, dev.num_sms, st)
               : launch_grouped_gemm(g1, Epilogue::kSwiGLU, dev.num_sms, st),
           "gate/up GEMM launch");
  MOE_CUDA(mark(4), "event record");
  MOE_CUDA(fp8 ? launch_grouped_gemm_2sm_fp8(g2, Epilogue::kScale, dev.num_sms, st)
               : launch_grouped_gemm(g2, Epilogue::kScale, dev.num_sms, st),
           "down GEMM launch");
  MOE_CUDA(mark(5), "event record");
  // stage 5: each token sums its k rows weighted by its TopK weights
  MOE_CUDA(launch_combine(y, dest_row, topk_w, T, k, d, out, &hdr->status, dev.num_sms, st), "combine launch");
  MOE_CUDA(mark(6), "event record");
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_forward(const void* x, const float* logits, const void* packed, int64_t T, int32_t d, int32_t E,
                         int32_t k, int32_t f, int32_t renormalize, void* out, int32_t* topk_idx_out,
                         float* topk_w_out, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  return forward_impl(x, logits, nullptr, packed, T, d, E, k, f, renormalize, out, topk_idx_out, topk_w_out,
                      workspace, workspace_bytes, stream, nullptr);
}

moe_status_t moe_forward_routed(const void* x, const void* router_packed, const void* packed, int64_t T, int32_t d,
                                int32_t E, int32_t k, int32_t f, int32_t renormalize, void* out,
                                int32_t* topk_idx_out, float* topk_w_out, void* workspace, size_t workspace_bytes,
                                moe_stream_t stream) {
  if (!router_packed) return fail(MOE_ERR_INVALID_ARG, "NULL router weights");
  return forward_impl(x, nullptr, router_packed, packed, T, d, E, k, f, renormalize, out, topk_idx_out, topk_w_out,
                      workspace, workspace_bytes, stream, nullptr);
}

moe_status_t moe_forward_timed(const void* x, const float* logits, const void* packed, int64_t T, int32_t d,
                               int32_t E, int32_t k, int32_t f, int32_t renormalize, void* out, void* workspace,
                               size_t workspace_bytes, moe_stream_t stream, void* const* events) {
  if (!events) return fail(MOE_ERR_INVALID_ARG, "NULL events");
  return forward_impl(x, logits, nullptr, packed, T, d, E, k, f, renormalize, out, nullptr, nullptr, workspace,
                      workspace_bytes, stream, events);
}

moe_status_t moe_forward_gathered(const void* x, const float* logits, const void* packed, int64_t T, int32_t d,
                                  int32_t E, int32_t k, int32_t f, int32_t renormalize, void* out,
                                  int32_t* topk_idx_out, float* topk_w_out, void* workspace, size_t workspace_bytes,
                                  moe_stream_t stream) {
  return forward_impl(x, logits, nullptr, packed, T, d, E, k, f, renormalize, out, topk_idx_out, topk_w_out,
                      workspace, workspace_bytes, stream, nullptr, true);
}

moe_status_t moe_forward_gathered_timed(const void* x, const float* logits, const void* packed, int64_t T, int32_t d,
                                        int32_t E, int32_t k, int32_t f, int32_t renormalize, void* out,
                                        void* workspace, size_t workspace_bytes, moe_stream_t stream,
                                        void* const* events) {
  if (!events) return fail(MOE_ERR_INVALID_ARG, "NULL events");
  return forward_impl(x, logits, nullptr, packed, T, d, E, k, f, renormalize, out, nullptr, nullptr, workspace,
                      workspace_bytes, stream, events, true);
}

size_t moe_fp8_packed_weight_bytes(int32_t E, int32_t d, int32_t f) {
  if (E < 1 || d < 128 || f < 128 || d % 128 != 0 || f % 128 != 0) return 0;
  return fp8_packed_bytes(E, d, f, nullptr);
}

moe_status_t moe_pack_weights_fp8(const uint8_t* gate_codes, const float* gate_scales, const uint8_t* up_codes,
                                  const float* up_scales, const uint8_t* down_codes, const float* down_scales,
                                  int32_t E, int32_t d, int32_t f, void* packed, moe_stream_t stream) {
  moe_status_t s = check_fp8_pack_dims(E, d, f);
  if (s != MOE_OK) return s;
  if (!gate_codes || !gate_scales || !up_codes || !up_scales || !down_codes || !down_scales || !packed)
    return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(gate_codes, 16) || !aligned(up_codes, 16) || !aligned(down_codes, 16) || !aligned(packed, kAlign))
    return fail(MOE_ERR_INVALID_ARG, "codes must be 16-byte and packed 256-byte aligned");
  if (!aligned(gate_scales, 4) || !aligned(up_scales, 4) || !aligned(down_scales, 4))
    return fail(MOE_ERR_INVALID_ARG, "scales must be 4-byte aligned");
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  MOE_CUDA(launch_pack_weights_fp8(gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, E, d, f,
                                   packed, dev.num_sms, static_cast<cudaStream_t>(stream)),
           "FP8 pack launch");
  return MOE_OK;
}

moe_status_t moe_forward_fp8(const void* x, const float* logits, const void* packed_fp8, int64_t T, int32_t d,
                             int32_t E, int32_t k, int32_t f, int32_t renormalize, void* out, int32_t* topk_idx_out,
                             float* topk_w_out, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  return forward_impl(x, logits, nullptr, packed_fp8, T, d, E, k, f, renormalize, out, topk_idx_out, topk_w_out,
                      workspace, workspace_bytes, stream, nullptr, false, true);
}

moe_status_t moe_forward_fp8_timed(const void* x, const float* logits, const void* packed_fp8, int64_t T, int32_t d,
                                   int32_t E, int32_t k, int32_t f, int32_t renormalize, void* out, void* workspace,
                                   size_t workspace_bytes, moe_stream_t stream, void* const* events) {
  if (!events) return fail(MOE_ERR_INVALID_ARG, "NULL events");
  return forward_impl(x, logits, nullptr, packed_fp8, T, d, E, k, f, renormalize, out, nullptr, nullptr, workspace,
                      workspace_bytes, stream, events, false, true);
}

moe_status_t moe_forward_host(const void* x_host, const float* logits_host, void* out_host, void* x_dev,
                              float* logits_dev, void* out_dev, const void* packed, int64_t T, int32_t d, int32_t E,
                              int32_t k, int32_t f, int32_t renormalize, void* workspace, size_t workspace_bytes,
                              moe_stream_t stream) {
  moe_status_t s = check_routing(T, E, k);
  if (s != MOE_OK) return s;
  if (T > 0 && (!x_host || !logits_host || !out_host || !x_dev || !logits_dev || !out_dev))
    return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t xb = static_cast<size_t>(T) * d * 2, lb = static_cast<size_t>(T) * E * 4;
  if (T > 0) {
    MOE_CUDA(cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, st), "x copy to device");
    MOE_CUDA(cudaMemcpyAsync(logits_dev, logits_host, lb, cudaMemcpyHostToDevice, st), "logits copy to device");
  }
  s = moe_forward(x_dev, logits_dev, packed, T, d, E, k, f, renormalize, out_dev, nullptr, nullptr, workspace,
                  workspace_bytes, stream);
  if (s != MOE_OK) return s;
  if (T > 0) MOE_CUDA(cudaMemcpyAsync(out_host, out_dev, xb, cudaMemcpyDeviceToHost, st), "out copy to host");
  MOE_CUDA(cudaStreamSynchronize(st), "stream synchronize");
  return MOE_OK;
}

moe_status_t moe_forward_host_stream(const void* const* x_host, const float* const* logits_host,
                                     void* const* out_host, int32_t n_batches, void* const* x_dev,
                                     float* const* logits_dev, void* const* out_dev, const void* packed, int64_t T,
                                     int32_t d, int32_t E, int32_t k, int32_t f, int32_t renormalize,
                                     void* workspace, size_t workspace_bytes, moe_stream_t stream,
                                     moe_stream_t copy_in, moe_stream_t copy_out) {
  moe_status_t s = check_routing(T, E, k);
  if (s != MOE_OK) return s;
  if (n_batches < 0) return fail(MOE_ERR_INVALID_ARG, "n_batches must be >= 0");
  if (n_batches == 0 || T == 0) return MOE_OK;
  if (!x_host || !logits_host || !out_host || !x_dev || !logits_dev || !out_dev)
    return fail(MOE_ERR_INVALID_ARG, "NULL pointer array");
  for (int b = 0; b < n_batches; ++b)
    if (!x_host[b] || !logits_host[b] || !out_host[b]) return fail(MOE_ERR_INVALID_ARG, "NULL host pointer");
  for (int i = 0; i < 2; ++i)
    if (!x_dev[i] || !logits_dev[i] || !out_dev[i]) return fail(MOE_ERR_INVALID_ARG, "NULL device slot");
  if (copy_in == stream || copy_out == stream || copy_in == copy_out)
    return fail(MOE_ERR_INVALID_ARG, "stream, copy_in and copy_out must be three different streams");
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaStream_t ci = static_cast<cudaStream_t>(copy_in);
  cudaStream_t co = static_cast<cudaStream_t>(copy_out);
  const size_t xb = static_cast<size_t>(T) * d * 2, lb = static_cast<size_t>(T) * E * 4;
  // per slot: inputs landed, compute done (slot inputs free, output ready), output copied (slot output free)
  cudaEvent_t ev[3][2] = {};
  moe_status_t result = MOE_OK;
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 3 && e == cudaSuccess; ++i)
    for (int j = 0; j < 2 && e == cudaSuccess; ++j) e = cudaEventCreateWithFlags(&ev[i][j], cudaEventDisableTiming);
  for (int b = 0; b < n_batches && e == cudaSuccess && result == MOE_OK; ++b) {
    const int sl = b & 1;
    if (b >= 2) e = cudaStreamWaitEvent(ci, ev[1][sl], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(x_dev[sl], x_host[b], xb, cudaMemcpyHostToDevice, ci);
    if (e == cudaSuccess) e = cudaMemcpyAsync(logits_dev[sl], logits_host[b], lb, cudaMemcpyHostToDevice, ci);
    if (e == cudaSuccess) e = cudaEventRecord(ev[0][sl], ci);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev[0][sl], 0);
    if (e == cudaSuccess && b >= 2) e = cudaStreamWaitEvent(cs, ev[2][sl], 0);
    if (e != cudaSuccess) break;
    result = moe_forward(x_dev[sl], logits_dev[sl], packed, T, d, E, k, f, renormalize, out_dev[sl], nullptr, nullptr,
                         workspace, workspace_bytes, stream);
    if (result != MOE_OK) break;
    e = cudaEventRecord(ev[1][sl], cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(co, ev[1][sl], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(out_host[b], out_dev[sl], xb, cudaMemcpyDeviceToHost, co);
    if (e == cudaSuccess) e = cudaEventRecord(ev[2][sl], co);
  }
  // whatever was enqueued completes before the events go away
  cudaError_t e2 = cudaStreamSynchronize(co);
  if (e2 == cudaSuccess) e2 = cudaStreamSynchronize(cs);
  if (e2 == cudaSuccess) e2 = cudaStreamSynchronize(ci);
  for (int i = 0; i < 3; ++i)
    for (int j = 0; j < 2; ++j)
      if (ev[i][j]) cudaEventDestroy(ev[i][j]);
  if (result != MOE_OK) return result;
  if (e != cudaSuccess) return cuda_fail(e, "pipelined host forward");
  if (e2 != cudaSuccess) return cuda_fail(e2, "stream synchronize");
  return MOE_OK;
}

size_t moe_backward_workspace_bytes(int64_t T, int32_t E, int32_t k, int32_t d, int32_t f) {
  if (T < 0 || E < 1 || k < 1 || d < 1 || f < 1) return 0;
  return backward_layout(T, E, k, d, f).total;
}

}  // extern "C"

namespace {

moe_status_t backward_impl(const void* x, const float* logits, const void* packed, const void* dout, int64_t T,
                           int32_t d, int32_t E, int32_t k, int32_t f, int32_t renormalize, void* dx,
                           float* d_logits, void* dw_gate, void* dw_up, void* dw_down, void* workspace,
                           size_t workspace_bytes, moe_stream_t stream, void* const* events) {
  moe_status_t s = check_routing(T, E, k);
  if (s != MOE_OK) return s;
  if ((s = check_gemm_dims(d, f)) != MOE_OK) return s;
  const int64_t P = T * k;
  if ((s = check_tile_space(P, E, d, f)) != MOE_OK) return s;
  if (static_cast<int64_t>(E) * ((std::max(d, f) + 127) / 128) * (2 * static_cast<int64_t>(f) / 64 + d / 64) >=
      (int64_t(1) << 31))
    return fail(MOE_ERR_UNSUPPORTED, "problem too large for the tile index");
  if (!packed || !dw_gate || !dw_up || !dw_down) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (T > 0 && (!x || !logits || !dout || !dx || !d_logits)) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  const void* al[] = {x, dout, dx, dw_gate, dw_up, dw_down, packed};
  for (const void* q : al)
    if (!aligned(q, 16)) return fail(MOE_ERR_INVALID_ARG, "x, dout, dx, the weight gradients and packed must be "
                                                          "16-byte aligned");
  const BackwardLayout L = backward_layout(T, E, k, d, f);
  if (!workspace || workspace_bytes < L.total || !aligned(workspace, kAlign))
    return fail(MOE_ERR_WORKSPACE, "backward workspace needs " + std::to_string(L.total) + " bytes, 256-byte aligned");
  DeviceInfo dev;
  if ((s = device_info(&dev)) != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  auto* hdr = reinterpret_cast<WsHeader*>(ws);
  const ForwardLayout& F = L.F;
  auto* hist = reinterpret_cast<int32_t*>(ws + F.hist);
  auto* counts = reinterpret_cast<int32_t*>(ws + F.counts);
  auto* offsets = reinterpret_cast<int32_t*>(ws + F.offsets);
  auto* topk_idx = reinterpret_cast<int32_t*>(ws + F.topk_idx);
  auto* topk_w = reinterpret_cast<float*>(ws + F.topk_w);
  auto* src_token = reinterpret_cast<int32_t*>(ws + F.src_token);
  auto* dest_row = reinterpret_cast<int32_t*>(ws + F.dest_row);
  auto* row_w = reinterpret_cast<float*>(ws + F.row_w);
  auto* d_topk_w = reinterpret_cast<float*>(ws + L.d_topk_w);
  void* x_perm = ws + F.x_perm;
  void* h = ws + F.h;
  void* y = ws + F.y;
  void* dx_perm = ws + F.y;  // y is dead by then (read by the output-reduction backward, or never written)
  void* gu = ws + L.gu;
  void* dy = ws + L.dy;
  void* dgu = ws + L.dgu;
  auto mark = [&](int i) -> cudaError_t {
    return events && events[i] ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) : cudaSuccess;
  };
  MOE_CUDA(mark(0), "event record");
  MOE_CUDA(cudaMemsetAsync(ws, 0, F.clear_bytes, st), "workspace clear");
  BackwardGemmArgs a{};
  a.P = P;
  a.E = E;
  a.d = d;
  a.f = f;
  a.offsets = offsets;
  a.w_gate_up = packed;
  a.w_down = static_cast<const __nv_bfloat16*>(packed) + static_cast<int64_t>(E) * 2 * f * d;
  a.x_perm = x_perm;
  a.dy = dy;
  a.h = h;
  a.gu = gu;
  a.dgu = dgu;
  a.dx_perm = dx_perm;
  a.dw_gate = dw_gate;
  a.dw_up = dw_up;
  a.dw_down = dw_down;
  a.counters = hdr->tile_counter;
  a.status = &hdr->status;
  if (T == 0) {
    // no rows: every weight gradient is zero
    MOE_CUDA(cudaMemsetAsync(offsets, 0, static_cast<size_t>(E + 1) * 4, st), "offsets clear");
    for (int i = 1; i <= 3; ++i) MOE_CUDA(mark(i), "event record");
    MOE_CUDA(launch_backward_dgrad_gemms(a, dev.num_sms, st, events ? events + 4 : nullptr), "dgrad GEMM launch");
    MOE_CUDA(mark(6), "event record");
    MOE_CUDA(launch_backward_wgrad_gemms(a, dev.num_sms, st, events ? events + 7 : nullptr), "wgrad GEMM launch");
    MOE_CUDA(mark(9), "event record");
    return MOE_OK;
  }
  // forward recomputation: stages 1-4 with G and U kept
  MOE_CUDA(launch_route_topk(logits, T, E, k, 1, renormalize, topk_idx, topk_w, hist, dev.num_sms, st),
           "route launch");
  MOE_CUDA(launch_index(topk_idx, topk_w, P, E, k, hist, counts, offsets, src_token, dest_row, row_w, &hdr->status,
                        st),
           "index launch");
  MOE_CUDA(launch_permute(x, T, d, dest_row, k, x_perm, &hdr->status, dev.num_sms, st), "permute launch");
  MOE_CUDA(mark(1), "event record");
  MOE_CUDA(launch_gate_up_save(a, dev.num_sms, st), "gate/up GEMM launch");
  MOE_CUDA(mark(2), "event record");
  if (backward_gate_grad_in_dgrad(E, d, f)) {
    // the down projection is not recomputed: the output gradient goes to
    // the rows as it is (dout_rows, in the dY buffer), the operand of the
    // dgrad down GEMM, which applies the gates itself and keeps its
    // accumulator before them in dh; the gate gradient <H, dh> then leaves
    // H gated in place, and the down weight gradient takes the gated H with
    // the ungated rows
    void* dout_rows = dy;
    void* dh = ws + L.dh;
    MOE_CUDA(launch_dout_permute(dout, dest_row, topk_w, T, k, d, dout_rows, nullptr, &hdr->status, dev.num_sms, st),
             "output-gradient permute launch");
    MOE_CUDA(mark(3), "event record");
    a.dy_dgrad = dout_rows;
    a.row_w = row_w;
    a.dh_raw = dh;
    a.h_wgrad = h;
    a.dy_wgrad = dout_rows;
    MOE_CUDA(launch_backward_dgrad_gemms(a, dev.num_sms, st, events ? events + 4 : nullptr), "dgrad GEMM launch");
    MOE_CUDA(launch_gate_grad(h, dh, dest_row, topk_w, T, k, f, d_topk_w, &hdr->status, dev.num_sms, st),
             "gate gradient launch");
    MOE_CUDA(launch_route_backward(logits, topk_idx, d_topk_w, T, E, k, renormalize, d_logits, dev.num_sms, st),
             "route backward launch");
    MOE_CUDA(mark(6), "event record");
    MOE_CUDA(launch_backward_wgrad_gemms(a, dev.num_sms, st, events ? events + 7 : nullptr), "wgrad GEMM launch");
  } else {
    // the down GEMM recomputed with ungated rows (the gates enter in the
    // output reduction), stage 5 backward, the gates back to the logits
    const auto* wdn = static_cast<const __nv_bfloat16*>(a.w_down);
    GroupedGemmProblem g2{h, wdn, offsets, nullptr, y, P, E, f, d, d, &hdr->tile_counter[1], &hdr->status};
    MOE_CUDA(launch_grouped_gemm(g2, Epilogue::kScale, dev.num_sms, st), "down GEMM launch");
    MOE_CUDA(launch_combine_backward(dout, y, dest_row, topk_w, T, k, d, dy, d_topk_w, &hdr->status, dev.num_sms,
                                     st),
             "combine backward launch");
    MOE_CUDA(launch_route_backward(logits, topk_idx, d_topk_w, T, E, k, renormalize, d_logits, dev.num_sms, st),
             "route backward launch");
    MOE_CUDA(mark(3), "event record");
    MOE_CUDA(launch_backward_dgrad_gemms(a, dev.num_sms, st, events ? events + 4 : nullptr), "dgrad GEMM launch");
    MOE_CUDA(mark(6), "event record");
    MOE_CUDA(launch_backward_wgrad_gemms(a, dev.num_sms, st, events ? events + 7 : nullptr), "wgrad GEMM launch");
  }
  // the transpose of the permute: each token sums its k row gradients
  MOE_CUDA(launch_combine(dx_perm, dest_row, nullptr, T, k, d, dx, &hdr->status, dev.num_sms, st), "un-permute launch");
  MOE_CUDA(mark(9), "event record");
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_backward(const void* x, const float* logits, const void* packed, const void* dout, int64_t T,
                          int32_t d, int32_t E, int32_t k, int32_t f, int32_t renormalize, void* dx, float* d_logits,
                          void* dw_gate, void* dw_up, void* dw_down, void* workspace, size_t workspace_bytes,
                          moe_stream_t stream) {
  return backward_impl(x, logits, packed, dout, T, d, E, k, f, renormalize, dx, d_logits, dw_gate, dw_up, dw_down,
                       workspace, workspace_bytes, stream, nullptr);
}

moe_status_t moe_backward_timed(const void* x, const float* logits, const void* packed, const void* dout, int64_t T,
                                int32_t d, int32_t E, int32_t k, int32_t f, int32_t renormalize, void* dx,
                                float* d_logits, void* dw_gate, void* dw_up, void* dw_down, void* workspace,
                                size_t workspace_bytes, moe_stream_t stream, void* const* events) {
  if (!events) return fail(MOE_ERR_INVALID_ARG, "NULL events");
  return backward_impl(x, logits, packed, dout, T, d, E, k, f, renormalize, dx, d_logits, dw_gate, dw_up, dw_down,
                       workspace, workspace_bytes, stream, events);
}

moe_status_t moe_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int64_t limit_ns,
                                       moe_stream_t stream) {
  if (limit_ns < 1 || limit_ns > static_cast<int64_t>(kWaitLimitNs))
    return fail(MOE_ERR_INVALID_ARG, "limit_ns must be in [1, 2e9]");
  if (!workspace || workspace_bytes < sizeof(WsHeader) || !aligned(workspace, kAlign))
    return fail(MOE_ERR_WORKSPACE, "workspace needs 256 bytes, 256-byte aligned");
  DeviceInfo dev;
  moe_status_t s = device_info(&dev);
  if (s != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_CUDA(cudaMemsetAsync(workspace, 0, sizeof(WsHeader), st), "workspace clear");
  MOE_CUDA(launch_wait_timeout(&static_cast<WsHeader*>(workspace)->status, static_cast<uint64_t>(limit_ns), st),
           "wait check launch");
  return MOE_OK;
}

moe_status_t moe_selftest_activation(const float* z, int64_t n, float* silu, float* sigmoid, moe_stream_t stream) {
  if (n < 0 || (n > 0 && (!z || !silu || !sigmoid))) return fail(MOE_ERR_INVALID_ARG, "bad n or NULL pointer");
  DeviceInfo dev;
  moe_status_t s = device_info(&dev);
  if (s != MOE_OK) return s;
  MOE_CUDA(launch_activation(z, n, silu, sigmoid, dev.num_sms, static_cast<cudaStream_t>(stream)),
           "activation launch");
  return MOE_OK;
}

moe_status_t moe_set_tile_schedule(int32_t mode) {
  if (mode != MOE_TILE_SCHEDULE_DYNAMIC && mode != MOE_TILE_SCHEDULE_STATIC)
    return fail(MOE_ERR_INVALID_ARG, "tile schedule must be MOE_TILE_SCHEDULE_DYNAMIC or MOE_TILE_SCHEDULE_STATIC");
  set_static_tile_schedule(mode == MOE_TILE_SCHEDULE_STATIC);
  return MOE_OK;
}

moe_status_t moe_occupy_sms(int32_t n_sms, int64_t duration_ns, moe_stream_t stream) {
  DeviceInfo dev;
  moe_status_t s = device_info(&dev);
  if (s != MOE_OK) return s;
  if (n_sms < 0 || n_sms > dev.num_sms) return fail(MOE_ERR_INVALID_ARG, "n_sms outside [0, the SM count]");
  if (duration_ns < 0 || duration_ns > 10000000000LL) return fail(MOE_ERR_INVALID_ARG, "duration_ns outside [0, 1e10]");
  MOE_CUDA(launch_occupy(n_sms, static_cast<uint64_t>(duration_ns), static_cast<cudaStream_t>(stream)),
           "occupy launch");
  return MOE_OK;
}

moe_status_t moe_read_device_status(const void* workspace, moe_stream_t stream, int32_t* status) {
  if (!workspace || !status) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  MOE_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "stream synchronize");
  MOE_CUDA(cudaMemcpy(status, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost), "status read");
  return MOE_OK;
}

moe_status_t moe_get_device_status(const void* workspace, moe_stream_t stream) {
  int32_t status = MOE_OK;
  const moe_status_t s = moe_read_device_status(workspace, stream, &status);
  if (s != MOE_OK) return s;
  if (status != MOE_OK) set_last_error(std::string("device status: ") + moe_status_string(static_cast<moe_status_t>(status)));
  return static_cast<moe_status_t>(status);
}

}  // extern "C"
