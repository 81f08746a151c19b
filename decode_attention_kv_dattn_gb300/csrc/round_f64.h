// One rounding from fp64 to the two narrow storage types the library writes:
// bf16 (the QK-normalised q and k, "pega-omni PR #4", the talker kernels:
// RoPE with QK-norm) and E4M3 (OCP FP8: 1 sign, 4 exponent bits with bias 7,
// 3 mantissa bits, no infinities, 0x7f = NaN, subnormals m * 2^-9; the fp8
// KV cache that "TensorFold PR #608" names and leaves out).
//
// Both take the fp64 bits apart and round the dropped mantissa bits to
// nearest, ties to even, so the result never passes through fp32. Plain C++
// apart from the qualifiers, so that the host test suite builds the same
// functions and checks them against the oracle's definitions.
#pragma once

#include <math.h>
#include <stdint.h>

#if !defined(DATTN_HD)
#if defined(__CUDACC__)
#define DATTN_HD __host__ __device__ __forceinline__
#else
#define DATTN_HD inline
#endif
#endif

namespace dattn {

DATTN_HD uint64_t f64_bits(double x) {
#if defined(__CUDA_ARCH__)
  return static_cast<uint64_t>(__double_as_longlong(x));
#else
  uint64_t b;
  __builtin_memcpy(&b, &x, 8);
  return b;
#endif
}

// The bf16 nearest to y (ties to even); magnitudes that round past the
// largest finite bf16 give infinity, a NaN gives the quiet NaN 0x7fc0.
DATTN_HD uint16_t bf16_from_f64(double y) {
  const uint64_t b = f64_bits(y);
  const uint16_t sign = static_cast<uint16_t>((b >> 48) & 0x8000u);
  const int e = static_cast<int>((b >> 52) & 0x7ff);
  const uint64_t m = b & 0xfffffffffffffull;
  if (e == 0x7ff) return m ? 0x7fc0 : static_cast<uint16_t>(sign | 0x7f80u);
  const double a = fabs(y);
  if (a < 0x1p-126) {
    // bf16 subnormals are the multiples of 2^-133 (a * 2^133 is exact, and
    // rint rounds it to nearest even); 128 of them is the smallest normal,
    // whose encoding is 128 as well
    const double q = rint(a * 0x1p133);
    return static_cast<uint16_t>(sign | static_cast<uint16_t>(q));
  }
  const uint32_t keep = static_cast<uint32_t>(m >> 45);
  const uint64_t rem = m & ((1ull << 45) - 1);
  uint32_t v = (static_cast<uint32_t>(e - 1023 + 127) << 7) | keep;
  if (rem > (1ull << 44) || (rem == (1ull << 44) && (keep & 1u))) ++v;
  if (v >= 0x7f80u) v = 0x7f80u;  // past the largest finite value: infinity
  return static_cast<uint16_t>(sign | v);
}

// The E4M3 byte nearest to y (ties to even), magnitudes past 448 - the
// largest finite value - saturating to 448; a NaN gives 0x7f.
DATTN_HD uint8_t e4m3_from_f64(double y) {
  if (isnan(y)) return 0x7f;
  const uint64_t b = f64_bits(y);
  const uint8_t sign = static_cast<uint8_t>((b >> 56) & 0x80u);
  const double a = fabs(y);
  if (a >= 448.0) return static_cast<uint8_t>(sign | 0x7eu);
  if (a < 0x1p-6) {
    // subnormals are the multiples of 2^-9; 8 of them is the smallest normal,
    // whose encoding is 8 as well
    return static_cast<uint8_t>(sign | static_cast<uint8_t>(rint(a * 0x1p9)));
  }
  const int e = static_cast<int>((b >> 52) & 0x7ff) - 1023;  // -6 .. 8
  const uint64_t m = b & 0xfffffffffffffull;
  const uint32_t keep = static_cast<uint32_t>(m >> 49);
  const uint64_t rem = m & ((1ull << 49) - 1);
  uint32_t v = (static_cast<uint32_t>(e + 7) << 3) | keep;
  if (rem > (1ull << 48) || (rem == (1ull << 48) && (keep & 1u))) ++v;
  if (v > 0x7eu) v = 0x7eu;
  return static_cast<uint8_t>(sign | v);
}

}  // namespace dattn
