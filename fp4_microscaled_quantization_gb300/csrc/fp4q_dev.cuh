// fp4q_dev.cuh -- device helpers of the GB300 quantizer kernels (sm_103a).
//
// Nothing here is shared with the CPU oracle; the arithmetic is re-derived
// from the format and algorithm definitions cited beside each helper.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp4q.h"

namespace fp4q {

// ---------------------------------------------------------------- Philox
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 32x32->64 multiplies with the multipliers 0xD2511F53 / 0xCD9E8D57, the key
// bumped by the Weyl constants 0x9E3779B9 / 0xBB67AE85 between rounds.
struct Philox4 {
  uint32_t v[4];
};

__host__ __device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    c1 = (uint32_t)p1;
    c3 = (uint32_t)p0;
    c0 = n0;
    c2 = n2;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  Philox4 o;
  o.v[0] = c0; o.v[1] = c1; o.v[2] = c2; o.v[3] = c3;
  return o;
}
// The ten rounds' keys of one seed, rk[2r] / rk[2r+1] for round r, made once
// on the host and passed in the kernel parameters, so that the kernels' rounds
// read them from the constant bank instead of bumping two keys per round.
inline void philox_round_keys(uint64_t seed, uint32_t (&rk)[20]) {
  uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    rk[2 * r] = k0;
    rk[2 * r + 1] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}
// philox4x32_10 with the round keys given.
__device__ __forceinline__ Philox4 philox4x32_10_rk(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                    const uint32_t (&rk)[20]) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ rk[2 * r];
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ rk[2 * r + 1];
    c1 = (uint32_t)p1;
    c3 = (uint32_t)p0;
    c0 = n0;
    c2 = n2;
  }
  Philox4 o;
  o.v[0] = c0; o.v[1] = c1; o.v[2] = c2; o.v[3] = c3;
  return o;
}

// ---------------------------------------------------------------- fp32 pairs
// Packed fp32 (FADD2/FMUL2/FFMA2 on sm_100-class SMs), each lane IEEE
// round-to-nearest, no contraction between separate calls.
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
// a - b as a + b * (-1): the product is exact, so one rounding, like a - b.
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// max(|a|, |b|) with NaN propagation; the sign of the result is meaningless.
__device__ __forceinline__ float absmax_nan(float a, float b) {
  float d;
  asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// ---------------------------------------------------------------- bf16
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// fp32 -> bf16 bits, round to nearest even (finite inputs).
__device__ __forceinline__ uint32_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

// ---------------------------------------------------------------- conversions
// Two fp32 -> one byte of two E2M1 codes, RTNE with saturation to +-6;
// `lo` lands in the low nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u16.u8 %0, t; }"
      : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight fp32 -> one word of eight E2M1 codes (element 0 in the low nibble).
__device__ __forceinline__ uint32_t cvt_e2m1x8(float v0, float v1, float v2, float v3, float v4,
                                               float v5, float v6, float v7) {
  uint32_t w;
  asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3}; }"
      : "=r"(w)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return w;
}

// fp32 >= 0 -> E4M3 byte, RTNE, saturating to 448 (satfinite).
__device__ __forceinline__ uint32_t cvt_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

// E4M3 byte -> fp32 (exact, through f16).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  uint32_t h2;
  uint16_t in = (uint16_t)(b & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// ---------------------------------------------------------------- status
__device__ __forceinline__ void raise_status(uint32_t* st, uint32_t bits) {
  if (st) atomicOr(st, bits);
}

// ---------------------------------------------------------------- layouts
// Byte offset of the scale of (row r, block k) in the MMA scale layout of a
// copy with nkb blocks per row (see FP4Q_SF_MMA in fp4q.h).
__device__ __forceinline__ int64_t sf_mma_offset(int64_t r, int64_t k, int64_t nkb) {
  return ((r >> 7) * (nkb >> 2) + (k >> 2)) * 512 + 16 * (r & 31) + 4 * ((r >> 5) & 3) + (k & 3);
}

}  // namespace fp4q
