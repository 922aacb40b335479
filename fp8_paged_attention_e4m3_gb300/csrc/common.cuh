// Device helpers shared by the sm_103a kernels of the verify-attention
// library: the exact E4M3 -> FP16 decode, asynchronous copies, tensor-core
// fragments and small math wrappers.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "params.h"

namespace vae4 {

// ---------------------------------------------------------------------------
// Exact E4M3 -> FP16 decode.
//
// An OCP E4M3FN byte is s.eeee.mmm with exponent bias 7; FP16 is
// s.eeeee.mmmmmmmmmm with bias 15.  Moving the 7 magnitude bits eeee.mmm
// into FP16 bits 13..7 (and the sign to bit 15) keeps the exponent field
// value e and the mantissa m, so the FP16 number is
//     normal:    2^(e-15) * (1 + m/8) = dec(b) * 2^-8
//     subnormal: 2^-14 * (m*128/1024) = m * 2^-17 = dec(b) * 2^-8
// i.e. exactly dec(b) * 2^-8 for every finite code (and +-0).  The factor
// 2^8 is folded into the FP32 scales applied to the accumulators.  The two
// NaN codes map to the finite 1.875 (480 * 2^-8); a decoded value is never
// NaN or infinite, so bytes that are later masked out cannot poison a sum.
// (The audited kernel decodes E4M3 exactly: PR #566 "[Kernel] Finalize the
// audited TP2 DFlash2 31/29 ms endpoint", Final audit.)
// ---------------------------------------------------------------------------
constexpr int kDecodeScaleLog2 = -8;

// Four E4M3 bytes (little-endian in w) -> two f16x2 words: lo = (b0, b1),
// hi = (b2, b3), each half holding dec(b) * 2^-8.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t &lo,
                                                uint32_t &hi) {
  // t = [b1:00:b0:00] -> each 16-bit half holds b << 8 = s<<15 | mag<<8;
  // subtracting (mag << 7) leaves s<<15 | mag<<7.
  const uint32_t t0 = __byte_perm(w, 0u, 0x1404);
  const uint32_t t1 = __byte_perm(w, 0u, 0x3424);
  lo = t0 - ((t0 >> 1) & 0x3F803F80u);
  hi = t1 - ((t1 >> 1) & 0x3F803F80u);
}

// Hardware converter: two E4M3 bytes -> f16x2, exact for every finite code
// (every E4M3 value is an FP16 value); byte 0 -> low half.  The two NaN
// codes become FP16 NaN.
__device__ __forceinline__ uint32_t cvt_e4m3x2(uint32_t two_bytes) {
  uint32_t d;
  const unsigned short v = (unsigned short)(two_bytes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(d) : "h"(v));
  return d;
}
// Four E4M3 bytes -> two f16x2 words (lo = bytes 0,1; hi = bytes 2,3), dec(b).
__device__ __forceinline__ void e4m3x4_to_f16x4_hw(uint32_t w, uint32_t &lo, uint32_t &hi) {
  lo = cvt_e4m3x2(w);
  hi = cvt_e4m3x2(w >> 16);
}
__device__ __forceinline__ void e4m3x16_to_f16x16_hw(const uint4 &raw, uint4 &h0, uint4 &h1) {
  e4m3x4_to_f16x4_hw(raw.x, h0.x, h0.y);
  e4m3x4_to_f16x4_hw(raw.y, h0.z, h0.w);
  e4m3x4_to_f16x4_hw(raw.z, h1.x, h1.y);
  e4m3x4_to_f16x4_hw(raw.w, h1.z, h1.w);
}

// Two FP8 bytes (byte 0 -> low half) -> f16x2, exact for every finite code.
// E4M3 through the hardware converter; an E5M2 byte is the high byte of the
// FP16 with the same value (same sign, 5-bit exponent with bias 15, the two
// mantissa bits on top of FP16's ten), so it is a byte move.
template <bool E5M2>
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint32_t two_bytes) {
  if constexpr (E5M2)
    return __byte_perm(two_bytes, 0u, 0x1404);  // (b1 << 24) | (b0 << 8)
  else
    return cvt_e4m3x2(two_bytes);
}

// 16 bytes -> 16 halves (two uint4 of f16x2).
__device__ __forceinline__ void e4m3x16_to_f16x16(const uint4 &raw, uint4 &h0,
                                                  uint4 &h1) {
  e4m3x4_to_f16x4(raw.x, h0.x, h0.y);
  e4m3x4_to_f16x4(raw.y, h0.z, h0.w);
  e4m3x4_to_f16x4(raw.z, h1.x, h1.y);
  e4m3x4_to_f16x4(raw.w, h1.z, h1.w);
}

// ---------------------------------------------------------------------------
// Asynchronous global -> shared copies (16 bytes, L2-only, zero fill).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src,
                                           bool valid) {
  const int n = valid ? 16 : 0;  // 0 bytes read -> 16 zero bytes written
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst),
               "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// Warp-level tensor-core fragments (m16n8k16, FP16 in, FP32 accumulate).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr));
}
// Two transposed 16 x 16 byte matrices (threads 0-15 give the 16 row
// addresses of the first, 16-31 of the second): thread i receives, of the
// first matrix, rows 4(i%4) .. 4(i%4)+3 of column i/4 in r[0] (row order
// = byte order) and of column i/4 + 8 in r[1]; r[2], r[3] likewise for
// the second matrix.
__device__ __forceinline__ void ldsm_b8_trans_x2(uint32_t (&r)[4], uint32_t addr) {
  asm volatile(
      "ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0,%1,%2,%3}, [%4];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr)
      : "memory");
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 2^x with the hardware approximation (relative error ~2^-22); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

}  // namespace vae4
