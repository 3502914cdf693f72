// Backward of the routing ends of the layer.
//
// combine_backward: "Scalable Pretraining of Large MoE LMs on Aurora Super
// Computer", §3.1, Algorithm 1, stage 5 (output reduction, backward): for
// every routed pair (t, j) at row r, mlp_out_grad[r] = w[t, j] *
// output_grad[t] and weights_grad[t, j] = <mlp_out[r], output_grad[t]>.
// One warp per token; each row's dot product sums in slot-independent
// lane order (the lane's pieces in order, then a butterfly over lanes).
//
// Without recomputing the expert outputs (the layer backward when the down
// projection's input gradient runs on SM pairs), stage 5's backward splits in
// two.  dout_permute writes each pair's row of the output gradient as it is
// (the operand of the down projection's input gradient, which applies the
// gate itself, and of the down weight gradient), and optionally gated
// (mlp_out_grad).  gate_grad forms weights_grad[t, j] = <mlp_out[r],
// output_grad[t]> as <H[r], dHu[r]>: with mlp_out[r] = H[r] Wd and dHu[r] =
// output_grad[t] Wd^T (that input gradient before the gate) it is the same
// product, summed in the other order; it then leaves H[r] gated in place,
// since H^T mlp_out_grad = (gated H)^T output_grad for the weight gradient.
//
// route_backward: the gates' gradient taken back to the router logits
// (Algorithm 1, stage 1, Softmax and TopK, with the selection held fixed):
// dl_e = [e is slot j] w_j dw_j - q_e * sum_j w_j dw_j, q the softmax over
// all E (or over the k selected when the gates are renormalised).  One warp
// per token holding the row's logits in registers.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kWarps = 8;

// The token's output-gradient row is read once: each lane walks its 16-byte
// pieces of that row and, for every piece, visits the k expert rows (their
// row index and gate broadcast from lane j), so a token's k rows are read
// and written once and dout is not re-read per slot.
template <int KMAX>
__global__ void __launch_bounds__(kWarps * 32)
combine_backward_kernel(const uint4* __restrict__ dout, const uint4* __restrict__ mlp_out,
                        const int32_t* __restrict__ dest_row, const float* __restrict__ w, int64_t T, int k, int dvec,
                        uint4* __restrict__ d_mlp_out, float* __restrict__ d_w, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t P = T * k;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); t < T; t += warps_total) {
    const int64_t my_row = lane < k ? __ldg(dest_row + t * k + lane) : 0;
    // a row outside [0, P) is never an address: that slot gets no row
    // gradient and a zero gate gradient
    const unsigned bad_slots = __ballot_sync(0xffffffffu, my_row < 0 || my_row >= P);
    if (bad_slots != 0u && lane == 0) record_status(status, kStatusBadIndex);
    const float my_w = lane < k ? __ldg(w + t * k + lane) : 0.f;
    const uint4* g = dout + t * dvec;
    float dot[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) dot[j] = 0.f;
    // the loop runs warp-uniformly (the shuffles need every lane); lanes past
    // the row's end take no load or store
    for (int v0 = 0; v0 < dvec; v0 += 32) {
      const int v = v0 + lane;
      const bool active = v < dvec;
      const uint4 gv = active ? __ldg(g + v) : make_uint4(0, 0, 0, 0);
      const __nv_bfloat162* gh = reinterpret_cast<const __nv_bfloat162*>(&gv);
      float2 gf[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) gf[i] = __bfloat1622float2(gh[i]);
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k) {
          const int64_t row = __shfl_sync(0xffffffffu, my_row, j);
          const float wj = __shfl_sync(0xffffffffu, my_w, j);
          if (active && !((bad_slots >> j) & 1u)) {
            const uint4 yv = __ldg(mlp_out + row * dvec + v);
            const __nv_bfloat162* yh = reinterpret_cast<const __nv_bfloat162*>(&yv);
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 yf = __bfloat1622float2(yh[i]);
              dot[j] = fmaf(yf.x, gf[i].x, dot[j]);
              dot[j] = fmaf(yf.y, gf[i].y, dot[j]);
              o[i] = pack_bf16x2(wj * gf[i].x, wj * gf[i].y);
            }
            d_mlp_out[row * dvec + v] = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        float s = dot[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) d_w[t * k + j] = s;
      }
    }
  }
}

// One warp per token: the token's output-gradient row is read once, piece
// by piece, and each piece written to its k rows as it is and (when gated is
// not null) scaled by the slot's gate.
template <int KMAX>
__global__ void __launch_bounds__(kWarps * 32)
dout_permute_kernel(const uint4* __restrict__ dout, const int32_t* __restrict__ dest_row, const float* __restrict__ w,
                    int64_t T, int k, int dvec, uint4* __restrict__ plain, uint4* __restrict__ gated, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t P = T * k;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); t < T; t += warps_total) {
    const int64_t my_row = lane < k ? __ldg(dest_row + t * k + lane) : 0;
    const unsigned bad_slots = __ballot_sync(0xffffffffu, my_row < 0 || my_row >= P);
    if (bad_slots != 0u && lane == 0) record_status(status, kStatusBadIndex);
    const float my_w = lane < k ? __ldg(w + t * k + lane) : 0.f;
    const uint4* g = dout + t * dvec;
    for (int v0 = 0; v0 < dvec; v0 += 32) {
      const int v = v0 + lane;
      const bool active = v < dvec;
      const uint4 gv = active ? __ldg(g + v) : make_uint4(0, 0, 0, 0);
      const __nv_bfloat162* gh = reinterpret_cast<const __nv_bfloat162*>(&gv);
      float2 gf[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) gf[i] = __bfloat1622float2(gh[i]);
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k) {
          const int64_t row = __shfl_sync(0xffffffffu, my_row, j);
          const float wj = __shfl_sync(0xffffffffu, my_w, j);
          if (active && !((bad_slots >> j) & 1u)) {
            plain[row * dvec + v] = gv;
            if (gated != nullptr) {
              uint32_t o[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) o[i] = pack_bf16x2(wj * gf[i].x, wj * gf[i].y);
              gated[row * dvec + v] = make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
        }
      }
    }
  }
}

// One warp per token: for each of its k rows, <h[r], dh_raw[r]> in fp32 --
// each lane its 16-byte pieces in order, then a butterfly over the lanes.
// With w not null each piece of h[r] is replaced, once read, by
// bf16(w[t, j] * h[r]): the gated rows the down weight gradient takes
// together with the ungated output-gradient rows.
__global__ void __launch_bounds__(kWarps * 32)
gate_grad_kernel(uint4* h, const uint4* __restrict__ dhu, const int32_t* __restrict__ dest_row,
                 const float* __restrict__ w, int64_t T, int k, int fvec, float* __restrict__ d_w, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t P = T * k;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); t < T; t += warps_total) {
    const int64_t my_row = lane < k ? __ldg(dest_row + t * k + lane) : 0;
    const unsigned bad_slots = __ballot_sync(0xffffffffu, my_row < 0 || my_row >= P);
    if (bad_slots != 0u && lane == 0) record_status(status, kStatusBadIndex);
    const float my_w = (w != nullptr && lane < k) ? __ldg(w + t * k + lane) : 0.f;
    for (int j = 0; j < k; ++j) {
      const int64_t row = __shfl_sync(0xffffffffu, my_row, j);
      const float wj = __shfl_sync(0xffffffffu, my_w, j);
      float s = 0.f;
      if (!((bad_slots >> j) & 1u)) {
        for (int v = lane; v < fvec; v += 32) {
          const uint4 hv = h[row * fvec + v];
          const uint4 dv = __ldg(dhu + row * fvec + v);
          const __nv_bfloat162* hh = reinterpret_cast<const __nv_bfloat162*>(&hv);
          const __nv_bfloat162* dh = reinterpret_cast<const __nv_bfloat162*>(&dv);
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 a = __bfloat1622float2(hh[i]);
            const float2 b = __bfloat1622float2(dh[i]);
            s = fmaf(a.x, b.x, s);
            s = fmaf(a.y, b.y, s);
            o[i] = pack_bf16x2(wj * a.x, wj * a.y);
          }
          if (w != nullptr) h[row * fvec + v] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) d_w[t * k + j] = s;
    }
  }
}

template <int NV>
__global__ void __launch_bounds__(kWarps * 32)
route_backward_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                      const float* __restrict__ d_w, int64_t T, int E, int k, int renormalize,
                      float* __restrict__ d_logits) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); t < T; t += warps_total) {
    const float* row = logits + t * E;
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = (lane + 32 * i < E) ? __ldg(row + lane + 32 * i) : -INFINITY;
    // lane j < k: slot j's expert, logit and gate gradient
    const int e_j = lane < k ? __ldg(idx + t * k + lane) : 0;
    const float l_j = lane < k ? __ldg(row + e_j) : -INFINITY;
    const float dw_j = lane < k ? __ldg(d_w + t * k + lane) : 0.f;
    // the normalisation set: all E experts, or the k selected
    float mx = renormalize ? l_j : -INFINITY;
    if (!renormalize) {
#pragma unroll
      for (int i = 0; i < NV; ++i) mx = fmaxf(mx, v[i]);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    float z = 0.f;
    if (renormalize) {
      z = lane < k ? expf(l_j - mx) : 0.f;
    } else {
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (lane + 32 * i < E) z += expf(v[i] - mx);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) z += __shfl_xor_sync(0xffffffffu, z, s);
    const float inv_z = 1.0f / __shfl_sync(0xffffffffu, z, 0);
    const float w_j = lane < k ? expf(l_j - mx) * inv_z : 0.f;
    float s_sum = w_j * dw_j;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) s_sum += __shfl_xor_sync(0xffffffffu, s_sum, s);
    s_sum = __shfl_sync(0xffffffffu, s_sum, 0);
    float g[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) g[i] = renormalize ? 0.f : -expf(v[i] - mx) * inv_z * s_sum;
    // slot j adds w_j dw_j (and, renormalised, its own -q s term) at its expert
    for (int j = 0; j < k; ++j) {
      const int e = __shfl_sync(0xffffffffu, e_j, j);
      const float add = __shfl_sync(0xffffffffu, renormalize ? w_j * (dw_j - s_sum) : w_j * dw_j, j);
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (lane + 32 * i == e) g[i] += add;
    }
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (lane + 32 * i < E) d_logits[t * E + lane + 32 * i] = g[i];
  }
}

// One token per warp up to 16 blocks per SM (two rounds of resident blocks):
// at 16k tokens each warp then takes one token and finished blocks make room
// for the rest, instead of every resident warp looping over 1-2 tokens.
int token_grid(int64_t T, int num_sms) {
  const int64_t want = (T + kWarps - 1) / kWarps;
  const int64_t cap = static_cast<int64_t>(num_sms) * 16;
  return static_cast<int>(want < cap ? want : cap);
}

}  // namespace

cudaError_t launch_combine_backward(const void* dout, const void* mlp_out, const int32_t* dest_row, const float* w,
                                    int64_t T, int k, int d, void* d_mlp_out, float* d_w, int32_t* status,
                                    int num_sms, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const auto* g = static_cast<const uint4*>(dout);
  const auto* y = static_cast<const uint4*>(mlp_out);
  auto* dy = static_cast<uint4*>(d_mlp_out);
  if (k <= 8)
    combine_backward_kernel<8><<<token_grid(T, num_sms), kWarps * 32, 0, stream>>>(g, y, dest_row, w, T, k, d / 8, dy,
                                                                                    d_w, status);
  else
    combine_backward_kernel<32><<<token_grid(T, num_sms), kWarps * 32, 0, stream>>>(g, y, dest_row, w, T, k, d / 8,
                                                                                     dy, d_w, status);
  return cudaGetLastError();
}

cudaError_t launch_dout_permute(const void* dout, const int32_t* dest_row, const float* w, int64_t T, int k, int d,
                                void* plain, void* gated, int32_t* status, int num_sms, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const auto* g = static_cast<const uint4*>(dout);
  auto* pl = static_cast<uint4*>(plain);
  auto* gt = static_cast<uint4*>(gated);
  if (k <= 8)
    dout_permute_kernel<8><<<token_grid(T, num_sms), kWarps * 32, 0, stream>>>(g, dest_row, w, T, k, d / 8, pl, gt,
                                                                                 status);
  else
    dout_permute_kernel<32><<<token_grid(T, num_sms), kWarps * 32, 0, stream>>>(g, dest_row, w, T, k, d / 8, pl, gt,
                                                                                  status);
  return cudaGetLastError();
}

cudaError_t launch_gate_grad(void* h, const void* dh_raw, const int32_t* dest_row, const float* w, int64_t T, int k,
                             int f, float* d_w, int32_t* status, int num_sms, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  gate_grad_kernel<<<token_grid(T, num_sms), kWarps * 32, 0, stream>>>(
      static_cast<uint4*>(h), static_cast<const uint4*>(dh_raw), dest_row, w, T, k, f / 8, d_w, status);
  return cudaGetLastError();
}

cudaError_t launch_route_backward(const float* logits, const int32_t* idx, const float* d_w, int64_t T, int E, int k,
                                  int renormalize, float* d_logits, int num_sms, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int grid = token_grid(T, num_sms);
  const int nv = (E + 31) / 32;
#define MOE_RB_CASE(NV)                                                                                           \
  route_backward_kernel<NV><<<grid, kWarps * 32, 0, stream>>>(logits, idx, d_w, T, E, k, renormalize, d_logits); \
  break;
  switch (nv <= 1 ? 1 : nv <= 2 ? 2 : nv <= 4 ? 4 : nv <= 8 ? 8 : nv <= 12 ? 12 : nv <= 16 ? 16 : 32) {
    case 1: MOE_RB_CASE(1)
    case 2: MOE_RB_CASE(2)
    case 4: MOE_RB_CASE(4)
    case 8: MOE_RB_CASE(8)
    case 12: MOE_RB_CASE(12)
    case 16: MOE_RB_CASE(16)
    default: MOE_RB_CASE(32)
  }
#undef MOE_RB_CASE
  return cudaGetLastError();
}

}  // namespace moe
