// fa4_exp2.cuh -- software 2^x on the FMA/ALU pipes, used beside MUFU.EX2.
//
// "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
// Asymmetric Hardware Scaling", §3.1.3 and Table 2: split 2^x into
// 2^floor(x) * 2^frac(x); the integer part is added to the IEEE-754
// exponent field with integer arithmetic (Cody-Waite style range
// reduction), the fractional part comes from a low-degree polynomial in
// Horner form on FMA units. Degree 3 suffices for BF16 probabilities.
//
// The pages do not print their coefficients. These are this library's own:
// the relative-error minimax fit of 1 + c1 f + c2 f^2 + c3 f^3 to 2^f on
// [0, 1] with the constant term held at exactly 1 (so 2^n is exact for
// integer n), found by the Remez exchange in fit_exp2_poly.py and rounded
// to fp32. Max relative error of the polynomial: 8.56e-5 (2^-13.5).
#pragma once
#include <cstdint>

namespace fa4 {

constexpr float kExp2C1 = 6.951167583e-01f;
constexpr float kExp2C2 = 2.276449949e-01f;
constexpr float kExp2C3 = 7.706703991e-02f;

// 2^x for x <= 128. Inputs are clamped to x >= -127; for x <= -126 the
// result is a value below 2^-126 (0 at x = -127), which plays the role of
// MUFU.EX2's flush to zero for softmax entries that small.
__device__ __forceinline__ float ex2_emulated(float x) {
  x = fmaxf(x, -127.0f);
  // Adding 1.5 * 2^23 with round-down leaves floor(x) in the low mantissa
  // bits of r (the fp32 spacing there is exactly 1).
  const float kShift = 12582912.0f;
  const float r = __fadd_rd(x, kShift);
  const float n = r - kShift;             // floor(x), exact
  const float f = x - n;                  // in [0, 1), exact
  const float poly = fmaf(fmaf(fmaf(kExp2C3, f, kExp2C2), f, kExp2C1), f, 1.0f);
  // (bits(r) << 23) == floor(x) << 23 modulo 2^32: the shifter's own bits
  // fall off the top, leaving the exponent increment.
  const uint32_t e = __float_as_uint(r) << 23;
  return __uint_as_float(__float_as_uint(poly) + e);
}

// The same computation on two inputs at once with the paired FP32
// instructions of sm_100+ (FFMA2 / FADD2): 6 instructions per element.
__device__ __forceinline__ float2 ex2_emulated2(float2 x) {
  const float2 kShift2 = make_float2(12582912.0f, 12582912.0f);
  const float2 kNegShift2 = make_float2(-12582912.0f, -12582912.0f);
  const float2 kMinusOne2 = make_float2(-1.0f, -1.0f);
  x.x = fmaxf(x.x, -127.0f);
  x.y = fmaxf(x.y, -127.0f);
  const float2 r = __fadd2_rd(x, kShift2);
  const float2 n = __fadd2_rn(r, kNegShift2);           // floor(x), exact
  const float2 f = __ffma2_rn(n, kMinusOne2, x);        // x - floor(x), exact
  float2 poly = __ffma2_rn(make_float2(kExp2C3, kExp2C3), f, make_float2(kExp2C2, kExp2C2));
  poly = __ffma2_rn(poly, f, make_float2(kExp2C1, kExp2C1));
  poly = __ffma2_rn(poly, f, make_float2(1.0f, 1.0f));
  return make_float2(__uint_as_float(__float_as_uint(poly.x) + (__float_as_uint(r.x) << 23)),
                     __uint_as_float(__float_as_uint(poly.y) + (__float_as_uint(r.y) << 23)));
}

}  // namespace fa4
