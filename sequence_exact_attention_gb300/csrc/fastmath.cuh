// Packed float32x2 arithmetic and a polynomial exp2 shared by the attention
// kernels (sm_100 family).
#pragma once

#include <cstdint>

#include "sm100.cuh"

namespace ra {
namespace fastmath {

// Three-input maximum (sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two float32 lanes packed in one 64-bit register: d = a * b + c, d = a + b.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fsub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// 2^x for two lanes on the FMA pipe, to take part of the exponentials off
// the special-function unit (which runs 16 ex2 per clock per SM, the
// bottleneck of the softmax otherwise). Cody-Waite style range reduction:
// x = n + f with n = round-to-nearest(x) taken from the low mantissa bits of
// x + 1.5*2^23, f = x - n in [-1/2, 1/2]; 2^f from a degree-3 polynomial
// fitted for minimum relative error on [-1/2, 1/2] with p(0) = 1 (relative
// error 1.02e-4, far below bf16's 2^-9 rounding of P); 2^n by adding n to
// the exponent field. x is clamped at -127, where the result is exactly +0
// (f = 0, p = 1, exponent 127 - 127), so masked scores still give 0.
constexpr float kExp2C1 = 6.932829022e-01f;
constexpr float kExp2C2 = 2.422103733e-01f;
constexpr float kExp2C3 = 5.500858277e-02f;
__device__ __forceinline__ void exp2_poly2(float x0, float x1, float& p0, float& p1) {
  const uint64_t magic = pack2(12582912.f, 12582912.f);
  const uint64_t x2 = pack2(fmaxf(x0, -127.f), fmaxf(x1, -127.f));
  const uint64_t t2 = fadd2(x2, magic);
  const uint64_t f2 = fsub2(x2, fsub2(t2, magic));
  uint64_t p2 = ffma2(pack2(kExp2C3, kExp2C3), f2, pack2(kExp2C2, kExp2C2));
  p2 = ffma2(p2, f2, pack2(kExp2C1, kExp2C1));
  p2 = ffma2(p2, f2, pack2(1.f, 1.f));
  float q0, q1, s0, s1;
  unpack2(p2, q0, q1);
  unpack2(t2, s0, s1);
  p0 = __uint_as_float(__float_as_uint(q0) + (__float_as_uint(s0) << 23));
  p1 = __uint_as_float(__float_as_uint(q1) + (__float_as_uint(s1) << 23));
}

}  // namespace fastmath
}  // namespace ra
