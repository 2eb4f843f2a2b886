// Exponentials for the softmax: the special-function unit's ex2.approx, and a polynomial
// form evaluated on the FMA and integer pipes.  The polynomial was built to move part of
// a row's exponentials off the special-function unit; in the forward it measured slower
// at both head dimensions on GB300 (d=64: 2.04 ms with every exponential on the unit,
// 2.31 ms with a quarter and 2.60 ms with half on the polynomial; d=128 with a quarter:
// 1.44 against 1.38 ms), because the softmax there is bound by instruction issue and its
// per-tile latency chain, and the polynomial costs about seven instructions per
// exponential against one.  The kernels therefore use ex2.approx; the polynomial stays
// available and tested (fa_selftest_exp2).
#pragma once

#include <cstdint>

#include "exp2_poly.h"
#include "sm100_ptx.cuh"

namespace fa {

// 2^x on the special-function unit (subnormal results flush to 0).
__device__ __forceinline__ float ex2_mufu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^x for two values at once, on the FMA and integer pipes only.  x = n + f with
// n = round(x) (adding 1.5 * 2^23 rounds to an integer and leaves n in the low mantissa
// bits) and f = x - n in [-1/2, 1/2]; 2^f comes from the polynomial of exp2_poly.h
// (relative error below 1.1e-4, exact at f = 0, so every integer x is exact), and 2^n is
// applied by adding n to the exponent field.  Valid for x <= 8 (2^8 = 256 is the largest value the softmax can
// produce); x < -125 (including -inf) gives exactly 0, like the flushed tiny results of
// ex2.approx.ftz.  Returns the two results packed as (lo, hi).
__device__ __forceinline__ uint64_t ex2_poly2(uint64_t x2) {
  constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
  const uint64_t t = fadd2(x2, f2pack(kRound, kRound));
  const uint64_t n = fadd2(t, f2pack(-kRound, -kRound));
  const uint64_t f = ffma2(n, f2pack(-1.0f, -1.0f), x2);
  uint64_t p = ffma2(f, f2pack(kExp2PolyC3, kExp2PolyC3), f2pack(kExp2PolyC2, kExp2PolyC2));
  p = ffma2(p, f, f2pack(kExp2PolyC1, kExp2PolyC1));
  p = ffma2(p, f, f2pack(1.0f, 1.0f));
  float p0, p1, t0, t1, x0, x1;
  f2unpack(p, p0, p1);
  f2unpack(t, t0, t1);
  f2unpack(x2, x0, x1);
  // the low 9 bits of 1.5 * 2^23's encoding are 0, so t's bits << 23 are n << 23
  float r0 = __int_as_float(__float_as_int(p0) + (__float_as_int(t0) << 23));
  float r1 = __int_as_float(__float_as_int(p1) + (__float_as_int(t1) << 23));
  r0 = x0 >= -125.0f ? r0 : 0.0f;
  r1 = x1 >= -125.0f ? r1 : 0.0f;
  return f2pack(r0, r1);
}

}  // namespace fa
