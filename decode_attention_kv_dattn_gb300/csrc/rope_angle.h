// RoPE angle: cos and sin of one rotary pair's angle at a position, from a
// 64-bit fixed-point phase and a short fp32 series.
//
// Plain C++ apart from the qualifiers, so that the host test suite can build
// the same function and check it against the exact values.
#pragma once

#include <stdint.h>

#include "bf16_exact.h"  // DATTN_HD, f32_mul, f32_fma

namespace dattn {

// int32 to fp32, rounded to nearest even.
DATTN_HD float f32_of_i32(int32_t x) {
#if defined(__CUDA_ARCH__)
  return __int2float_rn(x);
#else
  return static_cast<float>(x);  // the default rounding mode: to nearest, ties to even
#endif
}

// cos and sin of one RoPE pair's angle at position pos, as fp32 values.
// step = rint(2^64 * inv_freq / 2pi) is the pair's angle per position in
// 64-bit fixed-point turns, so pos * step mod 2^64 is the phase, exactly. Its
// top 32 bits split into a quadrant j (nearest quarter turn) and a remainder
// in [-1/8, 1/8) turn; cos and sin of the remainder t come from their Taylor
// series through t^10 and t^9 in fp32 (coefficients +-1/n!, first omitted
// terms below 2e-9 on [-pi/4, pi/4]) and are turned by j quarter turns. Every
// step is an integer or a correctly rounded fp32 operation (no contraction),
// so the result is the same on any IEEE machine: within 1.5e-7 of the exact
// values for |pos| <= 2^21, and no fp64 work.
DATTN_HD void rope_cos_sin(int64_t pos, uint64_t step, float& c, float& s) {
  const uint64_t phase = static_cast<uint64_t>(pos) * step;
  const uint32_t w = static_cast<uint32_t>(phase >> 32) + (1u << 29);
  const uint32_t quad = w >> 30;
  const int32_t rho = static_cast<int32_t>(w & 0x3fffffffu) - (1 << 29);
  const float t = f32_mul(f32_of_i32(rho), 1.46291807926715968e-09f);  // 2 pi / 2^32
  const float t2 = f32_mul(t, t);
  float sp = f32_fma(t2, 2.75573192e-06f, -1.98412698e-04f);
  sp = f32_fma(t2, sp, 8.33333333e-03f);
  sp = f32_fma(t2, sp, -1.66666667e-01f);
  const float sn = f32_fma(f32_mul(t, t2), sp, t);
  float cp = f32_fma(t2, -2.75573192e-07f, 2.48015873e-05f);
  cp = f32_fma(t2, cp, -1.38888889e-03f);
  cp = f32_fma(t2, cp, 4.16666667e-02f);
  cp = f32_fma(t2, cp, -5.0e-01f);
  const float cs = f32_fma(t2, cp, 1.0f);
  const float a = (quad & 1u) ? sn : cs;  // |cos| of the angle
  const float b = (quad & 1u) ? cs : sn;  // |sin| of the angle
  c = (quad == 1u || quad == 2u) ? -a : a;
  s = (quad >= 2u) ? -b : b;
}

}  // namespace dattn
