// Device helpers: inline PTX for mbarriers, TMA tile loads, ldmatrix, the
// warp-level bf16 / f16 MMA and the e4m3 conversions, plus bounded waits.
// Included by the kernel files only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "pa_internal.h"

namespace pa {

// A wait that has not completed after this many SM clocks (~0.2 s at 2 GHz;
// legitimate waits last microseconds) gives up, records PA_DEV_TIMEOUT and
// lets the kernel return.
constexpr long long kWaitBudget = 400000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void flag_status(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Returns false if the phase did not complete within the budget.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitBudget) return false;
  }
  return true;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// Byte offset of element (row, col) inside a [rows x 64] bf16 tile written by
// TMA with the 128-byte swizzle (16-byte chunk index XOR row % 8). The tile
// base must be 1024-byte aligned.
__device__ __forceinline__ uint32_t sw128(int row, int col) {
  return static_cast<uint32_t>(row * 128 + ((((col >> 3) ^ row) & 7) << 4) + ((col & 7) << 1));
}

// ---------------------------------------------------------------- warp MMA
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------- FP8 (e4m3)
// D += A(16x16, row) * B(16x8, col), f16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D += A(16x32, row) * B(32x8, col), e4m3 inputs (4 per register, lowest
// k-index in the lowest byte), fp32 accumulate. Every product is exact.
__device__ __forceinline__ void mma_16832_e4m3(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// f16x2 of two floats, lo in the low half (round to nearest even).
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// Two e4m3 bytes (low byte = element 0) to f16x2 (element 0 in the low
// half). Every e4m3 value is exact in f16.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  const __half2_raw h =
      __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_bytes), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}
// e4m3 bytes of two floats, lo in the low byte: round to nearest even,
// saturating to +-448 (NaN stays NaN).
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  return __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}
// Transpose of an 8x8 matrix of 16-bit elements held in the MMA fragment
// layout (lane i: row i / 4, elements 2 * (i % 4) and +1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(x));
  return d;
}
// Byte permute: bytes of {a, b} (a = bytes 0-3, b = 4-7) selected by sel.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Hardware base-2 exponential / logarithm (MUFU). ex2.approx of -inf is +0.
// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Element type of Q, the bf16/f16 K/V pools and the outputs: bfloat16
// (F16 = false) or IEEE half (F16 = true). Both are 2-byte types moved as raw
// bits; the kernels differ only in the MMA operand type and the conversions.
template <bool F16>
struct Elem;
template <>
struct Elem<false> {
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) { return pack_bf16(lo, hi); }
  static __device__ __forceinline__ float2 unpack(uint32_t v) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
  }
  static __device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
    mma_16816(d, a0, a1, a2, a3, b0, b1);
  }
  static constexpr uint32_t kTcFormat = 1;   // tcgen05 kind::f16 operand format: bf16
};
template <>
struct Elem<true> {
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) { return pack_f16(lo, hi); }
  static __device__ __forceinline__ float2 unpack(uint32_t v) {
    return __half22float2(*reinterpret_cast<const __half2*>(&v));
  }
  static __device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
    mma_16816_f16(d, a0, a1, a2, a3, b0, b1);
  }
  static constexpr uint32_t kTcFormat = 0;   // tcgen05 kind::f16 operand format: f16
};

// Two-lane float32 arithmetic (sm_100 and later): one instruction computes a
// pair, each lane rounded exactly as the scalar fmaf / add would be.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0,
                                      float b1, float c0, float c1) {
  asm("{\n\t.reg .b64 a, b, c, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1, float b0,
                                      float b1) {
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLog2e = 1.442695040888963407f;

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace pa

namespace pa {

// ---------------------------------------------------------------- tcgen05
// Tensor memory (TMEM) allocation, MMA issue/commit, and TMEM<->register
// moves. A warp may only touch TMEM lanes 32*(warp%4) .. +31.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, int ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, int ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f8f6f4 (e4m3 operands as
// the instruction descriptor's type fields say, fp32 accumulate; 32 bytes of
// K per instruction).
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]: A read from tensor memory (row m in
// lane m, two bf16 K-elements per 32-bit column), kind::f16.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                          uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Thread i of the warp writes 16 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// Thread i of the warp receives 32 consecutive 32-bit columns of lane
// (lane base + i), starting at column (taddr & 0xffff).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma: start address, leading
// and stride byte offsets (all >> 4), descriptor version 1 (bits 46-47) and
// the 128-byte swizzle layout (value 2 in bits 61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor for kind::f16 (and kind::f8f6f4) with fp32 D: D
// format (bits 4-5) = 1, A format (7-9) and B format (10-12) = fmt (kind::f16:
// 1 bf16, 0 f16; kind::f8f6f4: 0 e4m3; A and B of one MMA always share the
// type here), A K-major, B K-major or MN-major (bit 16), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N, bool b_mn_major, uint32_t fmt) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

}  // namespace pa

namespace pa {

// Programmatic dependent launch (griddepcontrol, sm_90 and later).
// pdl_wait: block until the grids this one depends on have completed and
// their writes are visible (a no-op for a grid launched without the
// attribute). pdl_trigger: allow the dependent grid to be scheduled once every
// block of this grid has executed it or exited.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ bool pdl_last_block() {
  return blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1;
}
// Entry of an attention kernel. The first kernel after the planner waits in
// every block (it reads the plan next) and only then lets the next kernel of
// the call be scheduled, so every later kernel starts with the plan complete.
// A later kernel lets its successor be scheduled at once and waits only in
// its last block, so that it cannot complete before its predecessor; the
// launchers size the grids one block past the last work item, so that this
// block has no work for the wait to delay.
__device__ __forceinline__ void pdl_enter(int pdl_first) {
  if (pdl_first) {
    pdl_wait();
    pdl_trigger();
  } else {
    pdl_trigger();
    if (pdl_last_block()) pdl_wait();
  }
}
// Exit of a kernel whose work does not depend on its predecessor (the K/V
// scatter): its last block waits at the end, after its own work, so that the
// grid still completes after its predecessor.
__device__ __forceinline__ void pdl_leave() {
  if (pdl_last_block()) pdl_wait();
}

// Fold a sink of logit s2 (base-2 units) into a row's final state kept as
// maximum m (base 2, -inf if no key was seen) and sum l relative to it: the
// new maximum is max(m, s2), the old sum (and the row's output, by the
// returned factor) are rescaled to it and 2^(s2 - max) joins the sum.
// Returns the factor for the unnormalised output; m and l are updated.
__device__ __forceinline__ float add_sink(float& m, float& l, float s2) {
  const float nm = fmaxf(m, s2);
  if (nm == -INFINITY) return 1.f;
  const float f = m == -INFINITY ? 0.f : fast_exp2(m - nm);
  l = l * f + fast_exp2(s2 - nm);
  m = nm;
  return f;
}

// A timeout anywhere in a launch sets the call's abort word; CTAs that start
// later see it and return at once, so a failing launch ends quickly.
__device__ __forceinline__ bool call_aborted(const AttnArgs& a) {
  return *reinterpret_cast<volatile const int*>(a.abort_all) != 0;
}
__device__ __forceinline__ void abort_call(const AttnArgs& a) {
  flag_status(a.status, PA_DEV_TIMEOUT);
  atomicExch(a.abort_all, 1);
}

// K/V producer shared by the attention kernels, run by one whole warp. Keys
// [kb, kb + ntiles*BN) of one KV head are loaded tile by tile into a ring of
// STAGES stages, each [K tile | V tile], each tile HALVES x [BN rows x 128 B]
// (128-byte swizzle). A tile is BN / box_rows TMA boxes per half; every box
// lies inside one page. The warp loads the page ids of the next 32 boxes
// (one per lane, coalesced) while the current ones are issued, so the
// block-table reads stay off the issue path; the boxes of a tile are issued
// by parallel lanes. A page id outside the pool, or
// a box past the sequence end, becomes the out-of-range coordinate
// num_blocks, which TMA fills with zeros. The unit's first tile is tile t0 of
// the ring's running sequence (stages and phases continue across units).
// SEP = false: one full/empty barrier pair per stage covers K and V, and
// issued[0] counts issued tiles. SEP = true: K and V of a stage have their own
// barriers -- full/empty[s] for K, full/empty[STAGES + s] for V -- so a
// consumer that is done with K(t) before V(t) can release it early, and
// issued[0] / issued[1] count the issued K / V tiles.
// Returns false on timeout/abort.
template <int BN, int HALVES, int STAGES, bool SEP = false>
__device__ bool produce_kv(const CUtensorMap* tmK, const CUtensorMap* tmV, const AttnArgs& a,
                           uint8_t* ring, uint64_t* full, uint64_t* empty,
                           volatile int* cta_abort, volatile int* issued,
                           const int32_t* bt_row, int hk, int kb, int kv_len, int ntiles,
                           int lane, int t0 = 0) {
  constexpr int HALF = BN * 128;
  constexpr int TILE = HALVES * HALF;
  constexpr int STAGE = 2 * TILE;
  const int box_rows = a.box_rows;
  const int bpt = BN / box_rows;         // boxes per tile
  const int tpg = 32 / bpt;              // tiles per group of 32 boxes
  const int ngroups = (ntiles + tpg - 1) / tpg;
  // Lane i holds the page id and page row of box i of a group.
  auto load_page = [&](int g, int& prow) -> int {
    const int k = kb + g * tpg * BN + lane * box_rows;
    int page = a.num_blocks;
    prow = 0;
    if (k < kv_len) {
      const int lp = k / a.bs;
      prow = k - lp * a.bs;
      const int pg = __ldg(bt_row + lp);
      if (pg >= 0 && pg < a.num_blocks) page = pg;
      else flag_status(a.status, PA_DEV_BAD_PAGE);
    }
    return page;
  };
  // The boxes of one tile are issued by parallel lanes: lane L takes box
  // L / (2*HALVES), half (L/2) % HALVES, K for even L and V for odd L.
  const int nbox = bpt * HALVES * 2;   // <= 32: box_rows >= 16, BN <= 128
  const int my_b = lane / (2 * HALVES), my_h = (lane >> 1) % HALVES, my_v = lane & 1;
  int next_row = 0, cur_row = 0;
  int next = ngroups > 0 ? load_page(0, next_row) : 0;
  for (int g = 0; g < ngroups; ++g) {
    const int cur = next;
    cur_row = next_row;
    if (g + 1 < ngroups) next = load_page(g + 1, next_row);
    for (int tt = 0; tt < tpg; ++tt) {
      const int t = g * tpg + tt;
      if (t >= ntiles) break;
      const int tr = t0 + t;   // position in the ring's sequence of tiles
      const int s = tr % STAGES;
      uint8_t* kdst = ring + s * STAGE;
      const int src = (tt * bpt + my_b) & 31;
      const int page = __shfl_sync(0xffffffffu, cur, src);
      const int prow = __shfl_sync(0xffffffffu, cur_row, src);
      // One pass per barrier pair: K and V together, or K then V.
#pragma unroll
      for (int part = 0; part < (SEP ? 2 : 1); ++part) {
        const int bi = SEP ? part * STAGES + s : s;
        int ok = 1;
        if (lane == 0) {
          if (tr >= STAGES && !mbar_wait(&empty[bi], ((tr / STAGES) - 1) & 1)) {
            abort_call(a);
            *cta_abort = 1;
          }
          if (*cta_abort) ok = 0;
          if (ok) mbar_arrive_expect_tx(&full[bi], SEP ? TILE : STAGE);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return false;
        if (lane < nbox && (!SEP || my_v == part))
          tma_load_4d(kdst + my_v * TILE + my_h * HALF + my_b * box_rows * 128, my_v ? tmV : tmK,
                      &full[bi], my_h * 64, hk, prow, page);
        if (lane == 0) issued[SEP ? part : 0] = tr + 1;
      }
    }
  }
  return true;
}

}  // namespace pa
