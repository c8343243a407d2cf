// Arithmetic shared by the page codecs (FP8 E4M3 and NVFP4): correctly rounded
// fp32 division without the division routine, packed fp32 pairs, and the
// absolute maximum of bf16 values.
//
// Every result here equals the IEEE fp32 operation it stands for, bit for bit;
// the codecs' tests compare codes and scales with a CPU implementation that
// performs the plain IEEE divisions.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace wa {
namespace codec {

// A divisor b for which the reciprocal r = RN(1/b) and every product below stay
// normal and finite: the range the Markstein sequence is used on.
__device__ __forceinline__ bool div_fast_ok(float b) { return b >= 1e-37f && b <= 1e37f; }

// A dividend a >= 0 that keeps a / c normal for the constants c used here
// (448, 2688): zero, or within [2^-100, 2^126].
__device__ __forceinline__ bool dividend_ok(float a) {
  return a == 0.f || (a >= 0x1p-100f && a <= 0x1p126f);
}

// RN(a / b) from r = RN(1 / b): q0 = RN(a r); the residual e = a - b q0 is
// exact in one FMA; q = RN(q0 + e r) is the correctly rounded quotient
// (Markstein's correction: P. Markstein, "Computation of elementary functions
// on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34 (1990)).  Valid
// for div_fast_ok(b) and a quotient that is zero or normal.
__device__ __forceinline__ float div_rn(float a, float b, float r) {
  const float q0 = __fmul_rn(a, r);
  const float e = __fmaf_rn(-b, q0, a);
  return __fmaf_rn(e, r, q0);
}

// Two fp32 lanes in one 64-bit register: {v, v}.
__device__ __forceinline__ uint64_t dup2(float v) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(v));
  return r;
}

// (q0, q1) = (RN(x0 / b), RN(x1 / b)) by the same sequence on packed lanes
// (mul.rn.f32x2, fma.rn.f32x2: each lane one IEEE operation), given
// nb2 = {-b, -b} and r2 = {RN(1/b), RN(1/b)}.  The sign of each quotient is set
// from its dividend: b > 0, so RN(x / b) has the sign of x, zeros included
// (the sequence alone returns +0 for x = -0).
__device__ __forceinline__ void div2_rn(float& q0, float& q1, float x0, float x1, uint64_t nb2,
                                        uint64_t r2) {
  asm("{\n\t.reg .b64 x, q, e;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mul.rn.f32x2 q, x, %5;\n\t"
      "fma.rn.f32x2 e, %4, q, x;\n\t"
      "fma.rn.f32x2 q, e, %5, q;\n\t"
      "mov.b64 {%0, %1}, q;\n\t}"
      : "=f"(q0), "=f"(q1)
      : "f"(x0), "f"(x1), "l"(nb2), "l"(r2));
  q0 = copysignf(q0, x0);
  q1 = copysignf(q1, x1);
}

// (d0, d1) = (a0 * b0, a1 * b1), one packed instruction, each RN
__device__ __forceinline__ void fmul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// two fp32 -> one bf16x2 word (RNE): lo in bits 0-15, hi in bits 16-31
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The two bf16 halves of w as fp32 (exact): lo = bits 0-15, hi = bits 16-31.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// max(|x|) over the 16 bf16 values of w[0..8), as fp32 (exact).  Pairs are
// combined with max.xorsign.abs.bf16x2, whose result has magnitude
// max(|a|, |b|) (its sign, the xor of the inputs' signs, is dropped at the end).
__device__ __forceinline__ float absmax16_bf16(const uint32_t (&w)[8]) {
  uint32_t m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[i]) : "r"(w[2 * i]), "r"(w[2 * i + 1]));
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[0]) : "r"(m[0]), "r"(m[1]));
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[2]) : "r"(m[2]), "r"(m[3]));
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[0]) : "r"(m[0]), "r"(m[2]));
  return fmaxf(__uint_as_float((m[0] & 0x7fffu) << 16), __uint_as_float(m[0] & 0x7fff0000u));
}

}  // namespace codec
}  // namespace wa
