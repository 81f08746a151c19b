// QK-norm of a head vector before RoPE ("pega-omni PR #4", the talker
// kernels: RoPE with QK-norm). The pages name the step but give no formula;
// the reading taken: per head, y_d = w_d * x_d / sqrt(mean(x^2) + eps) with one
// bf16 weight vector w [D] per layer for the queries and one for the keys,
// rounded once to bf16 (ties to even); RoPE then turns y as it would x.
//
// Arithmetic: the sum of squares, the root and the products in fp64. The
// square of a bf16 value is exact in fp64, so the sum is exact unless the
// squares span more than 2^37 in magnitude; y then lies within a few fp64
// ulps of its exact value, and its bf16 rounding is the exact value's except
// within that distance of a bf16 midpoint.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace dattn {

// The bf16 nearest to y (ties to even), in one rounding from fp64.
__device__ __forceinline__ uint16_t bf16_from_f64(double y) {
  const unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(y));
  const uint16_t sign = static_cast<uint16_t>((b >> 48) & 0x8000u);
  const int e = static_cast<int>((b >> 52) & 0x7ff);
  const unsigned long long m = b & 0xfffffffffffffull;
  if (e == 0x7ff) return m ? 0x7fc0 : static_cast<uint16_t>(sign | 0x7f80u);
  const double a = fabs(y);
  if (a < 0x1p-126) {
    // bf16 subnormals are the multiples of 2^-133; 128 of them is the
    // smallest normal, whose encoding is 128 as well
    const double q = rint(a * 0x1p133);
    return static_cast<uint16_t>(sign | static_cast<uint16_t>(q));
  }
  const uint32_t keep = static_cast<uint32_t>(m >> 45);
  const unsigned long long rem = m & ((1ull << 45) - 1);
  uint32_t v = (static_cast<uint32_t>(e - 1023 + 127) << 7) | keep;
  if (rem > (1ull << 44) || (rem == (1ull << 44) && (keep & 1u))) ++v;
  if (v >= 0x7f80u) v = 0x7f80u;  // past the largest finite value: infinity
  return static_cast<uint16_t>(sign | v);
}

// 1 / sqrt(mean(x^2) + eps) of one head vector x[0, D), by one warp: a
// lane-strided sum, then a butterfly, after which every lane holds the same
// bits (each level adds the same two values on both sides).
__device__ __forceinline__ double qk_norm_inv(const uint16_t* x, int D, double eps, int lane) {
  double ss = 0.0;
  for (int d = lane; d < D; d += 32) {
    const double v = bf16_to_f32(x[d]);
    ss = fma(v, v, ss);  // v * v is exact: fma and multiply-add agree
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  return 1.0 / sqrt(ss / D + eps);
}

// One normalised element: bf16(w * x * inv), the product taken left to right.
__device__ __forceinline__ uint16_t qk_norm_apply(uint16_t x, uint16_t w, double inv) {
  return bf16_from_f64(static_cast<double>(bf16_to_f32(w)) * static_cast<double>(bf16_to_f32(x)) * inv);
}

}  // namespace dattn
