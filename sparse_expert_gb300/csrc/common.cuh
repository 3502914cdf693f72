// Device-side helpers shared by the kernels of the MoE layer.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace moe {

// Device status codes (the values of moe_status_t in the public header).
enum : int32_t {
  kStatusOk = 0,
  kStatusTimeout = 4,
  kStatusBadIndex = 5,
};

// Every workspace starts with this header; one memset clears it per call.
struct WsHeader {
  int32_t status;          // first device error, or 0
  int32_t unused;
  int32_t tile_counter[6]; // persistent-GEMM tile counters (forward: gate/up, down;
                           // backward: dgrad down, dgrad gate/up, wgrad down, wgrad gate/up)
  int32_t reserved[56];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is one 256-byte line");

// Bound on every spin-wait in the kernels: far above any legitimate wait
// (microseconds), short enough that a broken pipeline ends the kernel.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, kStatusOk, code);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete.  Returns false when
// the wait ran out or another role of the block has given up (*abort != 0).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_addr(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// Same, taken by a whole warp with a warp-uniform outcome (needed before
// .sync.aligned instructions).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_addr(bar);
  uint64_t t0 = 0;
  const int lane = threadIdx.x & 31;
  if (lane == 0) t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    const bool ok = mbar_try_wait(a, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if ((it & 31u) == 31u) {
      int give_up = 0;
      if (lane == 0) give_up = (*abort != 0) || (global_timer_ns() - t0 > limit_ns);
      if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
    }
  }
}

// try_wait with a suspend-time hint: a thread whose phase is not complete is
// suspended until it completes or about hint_ns have passed, instead of
// returning at once, so a warp that waits long does not spin through the
// issue slots that the pipeline's producer and MMA threads need.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// mbar_wait_warp for long waits: the same bounded, warp-uniform outcome,
// each round suspending the warp for up to hint_ns.
__device__ __forceinline__ bool mbar_wait_warp_suspend(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                       uint32_t hint_ns = 20000, uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_addr(bar);
  uint64_t t0 = 0;
  const int lane = threadIdx.x & 31;
  if (lane == 0) t0 = global_timer_ns();
  for (;;) {
    const bool ok = mbar_try_wait_hint(a, parity, hint_ns);
    if (__all_sync(0xffffffffu, ok)) return true;
    int give_up = 0;
    if (lane == 0) give_up = (*abort != 0) || (global_timer_ns() - t0 > limit_ns);
    if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
  }
}

// ------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled bulk tensor load into shared memory, completion counted in bytes
// on `bar`.  c0 is the inner (contiguous) coordinate in elements.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, uint64_t* bar, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// 3-D tiled bulk tensor load (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(void* dst, const void* map, uint64_t* bar, int32_t c0, int32_t c1,
                                            int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::
          "r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Untiled bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global into this CTA's shared memory, completion counted in
// bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// --------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulator, one CTA.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// 32 TMEM lanes x 32 consecutive 32-bit columns; thread i of the warp gets
// lane (base lane + i).
__device__ __forceinline__ void tmem_ld_32x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 16 TMEM lanes x 32 consecutive 32-bit columns (four 16x256b blocks).
// Thread i gets lanes base + i/4 and base + 8 + i/4: r[4g] and r[4g + 1] are
// columns 8g + 2(i%4) and 8g + 2(i%4) + 1 of the first lane, r[4g + 2] and
// r[4g + 3] the same columns of the second.
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Four 8 x 8 bf16 matrices stored transposed: thread i holds in p_m the
// elements (row i/4, columns 2(i%4) and 2(i%4) + 1, low half first) of
// matrix m and gives the shared address of stored row i%8 of matrix i/8;
// stored row j of a matrix is its column j (16 bytes).
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t saddr, uint32_t p0, uint32_t p1, uint32_t p2,
                                                  uint32_t p3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(p0),
               "r"(p1), "r"(p2), "r"(p3)
               : "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// 128-byte swizzling: rows of 128 bytes, 8-row swizzle atoms of 1024 bytes
// stacked along M/N.  Fields: start address >> 4 (bits 0-13), leading byte
// offset (unused for this layout, 1), stride byte offset 1024 >> 4
// (bits 32-45), the fixed 0b001 of tcgen05 descriptors (bits 46-48), base
// offset 0 (tile bases are 1024-byte aligned), swizzle mode 2 = 128-byte
// (bits 61-63).  Moving along K inside the 128-byte row adds bytes >> 4 to
// the start address.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t desc = 0;
  desc |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  desc |= static_cast<uint64_t>(1) << 16;
  desc |= static_cast<uint64_t>(1024 >> 4) << 32;
  desc |= static_cast<uint64_t>(1) << 46;
  desc |= static_cast<uint64_t>(2) << 61;
  return desc;
}

// Shared-memory matrix descriptor of an MN-major bf16 operand written by TMA
// with 128-byte swizzling, as chunks of [K rows][64 MN values]: each K row
// of a chunk is 128 bytes (64 consecutive M or N indices), 8 K rows make a
// 1024-byte swizzle atom.  Stride byte offset (bits 32-45) = 1024 >> 4, the
// step between 8-row groups along K; leading byte offset (bits 16-29) =
// `chunk_bytes` >> 4, the step between 64-wide chunks along M or N.  Moving
// 16 rows along K (one MMA) adds 2048 bytes to the start address, so every
// start stays 1024-byte aligned (base offset 0).
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr, uint32_t chunk_bytes) {
  uint64_t desc = 0;
  desc |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  desc |= static_cast<uint64_t>((chunk_bytes >> 4) & 0x3FFFu) << 16;
  desc |= static_cast<uint64_t>(1024 >> 4) << 32;
  desc |= static_cast<uint64_t>(1) << 46;
  desc |= static_cast<uint64_t>(2) << 61;
  return desc;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A and B bf16 (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t umma_idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Same with the operands' major-ness: bit 15 set = A is MN-major (M
// contiguous), bit 16 set = B is MN-major (N contiguous).
__host__ __device__ constexpr uint32_t umma_idesc_bf16_f32_major(int M, int N, bool a_mn, bool b_mn) {
  return umma_idesc_bf16_f32(M, N) | (a_mn ? 1u << 15 : 0u) | (b_mn ? 1u << 16 : 0u);
}

// ------------------------------------------------------------------ misc
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// The hardware tanh (PTX tanh.approx.f32): one special-function operation.
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// sigmoid(z) = (1 + tanh(z / 2)) / 2 and Silu(z) = z sigmoid(z) = h + h tanh(h)
// with h = z / 2: one special-function operation each instead of an
// exponential and a reciprocal, which halves the epilogues' load on the
// special-function units.  Measured on GB300 against fp64 over [-20, 20]
// (moe_selftest_activation): sigmoid within 4e-6 absolute, Silu within 1e-5
// absolute and 1e-4 relative for z >= -4, within one bf16 ulp for z >= -8;
// below that Silu is smaller than 3e-3 and its absolute error stays below
// 1e-5 (the tanh saturates at -1 and the result reaches exactly 0).
__device__ __forceinline__ float sigmoid_f32(float z) { return fmaf(0.5f, tanh_approx(0.5f * z), 0.5f); }
__device__ __forceinline__ float silu_f32(float z) {
  const float h = 0.5f * z;
  return fmaf(h, tanh_approx(h), h);
}

}  // namespace moe
