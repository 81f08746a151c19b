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
#include "round_f64.h"

namespace dattn {

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
