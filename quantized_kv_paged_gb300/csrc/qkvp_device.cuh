// Device helpers of libqkvp: number-format conversions and thin PTX wrappers for sm_103a.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace qkvp {
namespace dev {

// ---------------------------------------------------------------------------------------------
// Encoders (quantize-on-append). Rounding is the hardware's round-to-nearest-even with
// saturation to the largest finite value; sign and NaN handling are made explicit here so that
// they do not depend on how the conversion instruction treats them:
//   E4M3: |x| >= 448 (and inf) -> 448; NaN -> 0x7F; the sign bit always follows x.
//   E2M1: |x| >= 6 -> 6; NaN -> 0x0; the sign bit always follows x (so -0.1 -> 0x8).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cvt_e4m3_satfinite(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;  // the second source lands in the low byte
}

__device__ __forceinline__ uint32_t encode_e4m3(float x) {
  if (x != x) return 0x7Fu;
  const uint32_t sign = (__float_as_uint(x) >> 24) & 0x80u;
  return sign | (cvt_e4m3_satfinite(fabsf(x)) & 0x7Fu);
}

__device__ __forceinline__ uint32_t cvt_e2m1_satfinite(float x) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r) : "f"(0.0f), "f"(x));
  return r & 0xFu;   // the second source lands in the low nibble
}

__device__ __forceinline__ uint32_t encode_e2m1(float x) {
  if (x != x) return 0x0u;
  const uint32_t sign = (__float_as_uint(x) >> 28) & 0x8u;
  return sign | (cvt_e2m1_satfinite(fabsf(x)) & 0x7u);
}

// ---------------------------------------------------------------------------------------------
// Decoders to FP16, the tensor-core operand type of the decode kernels. E4M3 -> F16 and E2M1 -> F16
// are exact hardware conversions (every E4M3 and E2M1 value is a normal F16); the NVFP4 product
// e2m1 * block scale has at most 6 significant bits and lies in [2^-10, 2688], so the F16 multiply
// is exact too.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
  return r;  // low half <- low byte
}

__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.u8.u32 t, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(r) : "r"(byte));
  return r;  // low half <- low nibble
}

// F16x2 -> E4M3x2 (low byte <- low half), round to nearest even, saturating to +-448.
__device__ __forceinline__ uint32_t f16x2_to_e4m3x2(uint32_t h2) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h2));
  return r;
}

// Two FP32 -> E4M3x2 (low byte <- lo), round to nearest even, saturating to +-448.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// The four code pairs of a 32-bit word (byte k = codes 2k, 2k + 1) -> four F16x2, exact: the word is
// unpacked into byte registers, so no per-byte shift or mask is needed.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}

__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  const uint32_t h2 = e4m3x2_to_f16x2(static_cast<uint16_t>(byte & 0xFFu));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// Two floats -> F16x2 (low half = lo), round to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two BF16 (low half = first) -> F16x2; exact for values within the F16 normal range.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t two, float scale = 1.0f) {
  return pack_f16x2(__uint_as_float(two << 16) * scale, __uint_as_float(two & 0xFFFF0000u) * scale);
}

// One packed NVFP4 byte (low nibble = first element) times a block scale held as F16x2 (both
// halves equal) -> F16x2, exact.
__device__ __forceinline__ uint32_t nvfp4x2_to_f16x2(uint32_t byte, uint32_t scale_h2) {
  return hmul2_f16(e2m1x2_to_f16x2(byte), scale_h2);
}

// E4M3 pair -> BF16 pair, exact (for the pool-wide cast of the cast-then-attend baseline).
__device__ __forceinline__ uint32_t fp8x2_to_bf16x2(uint32_t two) {
  const uint32_t h2 = e4m3x2_to_f16x2(static_cast<uint16_t>(two & 0xFFFFu));
  uint16_t lo, hi;
  asm("cvt.rn.bf16.f16 %0, %1;" : "=h"(lo) : "h"(static_cast<uint16_t>(h2 & 0xFFFFu)));
  asm("cvt.rn.bf16.f16 %0, %1;" : "=h"(hi) : "h"(static_cast<uint16_t>(h2 >> 16)));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// ---------------------------------------------------------------------------------------------
// Async copies and warp-level MMA (the mma.sync kernel).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x1(uint32_t addr, uint32_t& r0) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x1.shared.b16 {%0}, [%1];" : "=r"(r0) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
// Two 16x16 byte matrices, transposed (lanes 0..15 address the rows of the first, 16..31 of the
// second): lane l receives, of each matrix, rows 4(l%4) .. 4(l%4)+3 of column l/4 (one register, row
// 4(l%4) in the low byte) and of column 8 + l/4 (the next register). Checked on GB300.
__device__ __forceinline__ void ldsm_t8_x2(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// D += A * B, m16n8k16, F16 inputs, FP32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {  // round to nearest even
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

}  // namespace dev
}  // namespace qkvp
