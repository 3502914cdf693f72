// moe_dispatch_scan_noalloc: the counts / offsets / index pass of
// moe_dispatch_scan for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a scratch buffer at call
// time: inference-engine plugins and framework extensions whose host owns
// every device allocation and passes only the input and output tensors to
// the enqueue call, and latency-critical loops that must not call
// cudaMalloc (it can synchronise the device, and under memory pressure it
// can fail in the middle of a run).  For them, the scratch of the dispatch
// pass (status word and the per-chunk count table) lives in a fixed device
// array compiled into the library.
//
// The array is kStaticScratchBytes (4 MiB) per GPU and every GPU that loads
// the library keeps it until the process exits.  All calls share it and it
// keeps the previous call's contents, so each call clears the part that
// must start at zero; calls that overlap on the GPU (two streams, or two
// host threads on one device) race on it and must be serialised by the
// caller.  The first call on a device looks up the array's device address
// (cudaGetSymbolAddress) with that device current; make that first call
// before any stream capture.  The call itself allocates nothing: no
// cudaMalloc, no cudaFree, no allocating library routine.
//
// Errors the kernels find (an expert index outside [0, E)) land in the
// status word at the start of the array, which the next call clears;
// moe_dispatch_noalloc_status reads it back.
#include <mutex>
#include <string>

#include "moe_gb300.h"
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_dispatch_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_dispatch_scratch on the current device, looked up
// once per device.  In host code the array's name is only a host-side
// handle; kernels must be given this address instead.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

moe_status_t noalloc_fail(moe_status_t s, const std::string& msg) {
  set_last_error(msg);
  return s;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_dispatch_scan_noalloc(const int32_t* topk_idx, const float* topk_w, int64_t T,
                                                  int32_t E, int32_t k, int32_t* counts, int32_t* offsets,
                                                  int32_t* src_token, int32_t* dest_row, float* row_w,
                                                  moe_stream_t stream) {
  const moe_status_t checked = check_routing(T, E, k);
  if (checked != MOE_OK) return checked;
  if (!counts || !offsets) return noalloc_fail(MOE_ERR_INVALID_ARG, "NULL counts/offsets");
  if (T > 0 && (!topk_idx || !src_token || !dest_row)) return noalloc_fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (row_w && !topk_w) return noalloc_fail(MOE_ERR_INVALID_ARG, "row_w needs topk_w");
  const int64_t P = T * k;
  const size_t need = sizeof(WsHeader) + dispatch_hist_bytes(P, E);
  if (need > kStaticScratchBytes)
    return noalloc_fail(MOE_ERR_UNSUPPORTED,
                        "this problem needs " + std::to_string(need) + " bytes of scratch; the static scratch of "
                        "moe_dispatch_scan_noalloc holds " + std::to_string(kStaticScratchBytes) +
                        " bytes (use moe_dispatch_scan with a workspace)");
  DeviceInfo dev;
  cudaError_t e = current_device_info(&dev);
  if (e != cudaSuccess) return noalloc_fail(MOE_ERR_NO_DEVICE, std::string("device query: ") + cudaGetErrorName(e));
  if (dev.cc_major != 10 || dev.cc_minor != 3)
    return noalloc_fail(MOE_ERR_NO_DEVICE, "the library is built for sm_103a (GB300)");
  void* ws = nullptr;
  if ((e = scratch_address(&ws)) != cudaSuccess)
    return noalloc_fail(MOE_ERR_CUDA, std::string("static scratch address: ") + cudaGetErrorName(e));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the header (status word) must start at zero; the histogram kernel writes
  // every row of the count table
  if ((e = cudaMemsetAsync(ws, 0, sizeof(WsHeader), st)) != cudaSuccess)
    return noalloc_fail(MOE_ERR_CUDA, std::string("scratch clear: ") + cudaGetErrorName(e));
  if (P == 0) {
    if ((e = cudaMemsetAsync(counts, 0, static_cast<size_t>(E) * 4, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(offsets, 0, static_cast<size_t>(E + 1) * 4, st)) != cudaSuccess)
      return noalloc_fail(MOE_ERR_CUDA, std::string("counts/offsets clear: ") + cudaGetErrorName(e));
    return MOE_OK;
  }
  auto* hdr = static_cast<WsHeader*>(ws);
  auto* hist = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + sizeof(WsHeader));
  if ((e = launch_chunk_histogram(topk_idx, P, E, hist, &hdr->status, st)) != cudaSuccess)
    return noalloc_fail(MOE_ERR_CUDA, std::string("histogram launch: ") + cudaGetErrorName(e));
  if ((e = launch_index(topk_idx, topk_w, P, E, k, hist, counts, offsets, src_token, dest_row, row_w, &hdr->status,
                        st)) != cudaSuccess)
    return noalloc_fail(MOE_ERR_CUDA, std::string("index launch: ") + cudaGetErrorName(e));
  return MOE_OK;
}

extern "C" moe_status_t moe_dispatch_noalloc_status(moe_stream_t stream, int32_t* status) {
  if (!status) return noalloc_fail(MOE_ERR_INVALID_ARG, "NULL status");
  void* ws = nullptr;
  cudaError_t e = scratch_address(&ws);
  if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver)
    return noalloc_fail(MOE_ERR_NO_DEVICE, "no CUDA device available");
  if (e != cudaSuccess) return noalloc_fail(MOE_ERR_CUDA, std::string("static scratch address: ") + cudaGetErrorName(e));
  if ((e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return noalloc_fail(MOE_ERR_CUDA, std::string("stream synchronize: ") + cudaGetErrorName(e));
  // the header's status word, copied straight into the caller's int (no staging buffer)
  if ((e = cudaMemcpy(status, &static_cast<const WsHeader*>(ws)->status, sizeof(int32_t), cudaMemcpyDeviceToHost)) !=
      cudaSuccess)
    return noalloc_fail(MOE_ERR_CUDA, std::string("status read: ") + cudaGetErrorName(e));
  return MOE_OK;
}
