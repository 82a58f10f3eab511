// 2^x on the FMA pipe, two values at a time (packed fp32x2), to share the softmax's
// exponentials between the special-function unit (ex2.approx) and the FMA units.
//
//   2^x = 2^n * 2^f,  n = round(x),  f = x - n in [-1/2, 1/2]    (Cody-Waite range reduction)
//   2^f ~ c0 + c1 f + c2 f^2 + c3 f^3 + c4 f^4                    (minimax relative error)
// n is obtained by adding 1.5 * 2^23 (the integer lands in the low mantissa bits of the sum)
// and 2^n is applied by adding n << 23 to the bits of the polynomial's value.
// The coefficients are the degree-4 Remez fit printed by gen_exp2_poly.py (max relative
// error 2.6e-6 with fp32 coefficients). Inputs are clamped to >= -125, so results are
// >= 2^-125.5 (normal floats); inputs must be <= 126.
#pragma once

#include <cstdint>

namespace dit {

__device__ __forceinline__ void exp2_fma2(float& y0, float& y1, float x0, float x1) {
  constexpr float kShift = 12582912.0f;              // 1.5 * 2^23
  constexpr float c0 = 0.9999992847442627f, c1 = 0.6931217908859253f, c2 = 0.240247443318367f,
                  c3 = 0.05591785907745361f, c4 = 0.009570102207362652f;
  x0 = fmaxf(x0, -125.0f);
  x1 = fmaxf(x1, -125.0f);
  uint32_t t0, t1;
  float p0, p1;
  asm("{\n\t.reg .b64 X, T, R, F, P, C;\n\t"
      "mov.b64 X, {%4, %5};\n\t"
      "mov.b64 C, {%6, %6};\n\t"
      "add.rn.f32x2 T, X, C;\n\t"                     // T = x + 1.5*2^23 (round to nearest)
      "sub.rn.f32x2 R, T, C;\n\t"                     // R = n
      "sub.rn.f32x2 F, X, R;\n\t"                     // F = x - n
      "mov.b64 P, {%7, %7};\n\t"
      "mov.b64 C, {%8, %8};\n\t"
      "fma.rn.f32x2 P, P, F, C;\n\t"
      "mov.b64 C, {%9, %9};\n\t"
      "fma.rn.f32x2 P, P, F, C;\n\t"
      "mov.b64 C, {%10, %10};\n\t"
      "fma.rn.f32x2 P, P, F, C;\n\t"
      "mov.b64 C, {%11, %11};\n\t"
      "fma.rn.f32x2 P, P, F, C;\n\t"
      "mov.b64 {%0, %1}, T;\n\t"
      "mov.b64 {%2, %3}, P;\n\t}"
      : "=r"(t0), "=r"(t1), "=f"(p0), "=f"(p1)
      : "f"(x0), "f"(x1), "f"(kShift), "f"(c4), "f"(c3), "f"(c2), "f"(c1), "f"(c0));
  y0 = __uint_as_float(__float_as_uint(p0) + (t0 << 23));
  y1 = __uint_as_float(__float_as_uint(p1) + (t1 << 23));
}

}  // namespace dit
