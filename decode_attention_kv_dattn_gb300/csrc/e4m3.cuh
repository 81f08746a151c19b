// E4M3 (OCP FP8: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
// infinities, 0x7f = NaN, subnormals m * 2^-9) for fp8 KV caches: a cached
// value is e4m3 * scale, one scale per layer for K and one for V.
#pragma once

#include <cstdint>

namespace dattn {

// The E4M3 byte nearest to y (ties to even), magnitudes past 448 - the
// largest finite value - saturating to 448; one rounding from fp64.
__device__ __forceinline__ uint8_t e4m3_from_f64(double y) {
  if (isnan(y)) return 0x7f;
  const unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(y));
  const uint8_t sign = static_cast<uint8_t>((b >> 56) & 0x80u);
  const double a = fabs(y);
  if (a >= 448.0) return static_cast<uint8_t>(sign | 0x7eu);
  if (a < 0x1p-6) {
    // subnormals are the multiples of 2^-9; 8 of them is the smallest normal,
    // whose encoding is 8 as well
    return static_cast<uint8_t>(sign | static_cast<uint8_t>(rint(a * 0x1p9)));
  }
  const int e = static_cast<int>((b >> 52) & 0x7ff) - 1023;  // -6 .. 8
  const unsigned long long m = b & 0xfffffffffffffull;
  const uint32_t keep = static_cast<uint32_t>(m >> 49);
  const unsigned long long rem = m & ((1ull << 49) - 1);
  uint32_t v = (static_cast<uint32_t>(e + 7) << 3) | keep;
  if (rem > (1ull << 48) || (rem == (1ull << 48) && (keep & 1u))) ++v;
  if (v > 0x7eu) v = 0x7eu;
  return static_cast<uint8_t>(sign | v);
}

}  // namespace dattn
