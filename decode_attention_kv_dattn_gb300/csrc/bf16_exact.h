// Exact rounding of a rotated key element to bf16, in integer arithmetic.
//
// The K entry of RoPE (rotate-half, "vllm-omni commits", Spark model commit)
// is x*c + y*s for bf16 x, y and fp32 c, s (the pair's cos and sin, or -sin).
// Each product has at most 8 + 24 = 32 significant bits, so the exact sum is
// a 64-bit integer times a power of two whenever the two exponents are within
// 30 of each other; otherwise the smaller product lies wholly below the bits
// that the result can keep and only says which way an exact tie would go,
// which rounding to odd at integer precision records. The result is the
// bf16 nearest to the exact value, ties to even - no intermediate rounding,
// and no fp64 arithmetic (whose rate on this GPU is a small fraction of the
// integer pipes').
//
// Plain C++ apart from the qualifiers, so that the host test suite can build
// the same function and check it against the definition.
#pragma once

#include <stdint.h>

#if !defined(DATTN_HD)
#if defined(__CUDACC__)
#define DATTN_HD __host__ __device__ __forceinline__
#else
#define DATTN_HD inline
#endif
#endif

namespace dattn {

DATTN_HD int clz64_portable(uint64_t v) {
#if defined(__CUDA_ARCH__)
  return __clzll(static_cast<long long>(v));
#else
  return v == 0 ? 64 : __builtin_clzll(v);
#endif
}

// bf16 bits of the nearest value to x*c + y*s (x, y: bf16 bit patterns; c, s:
// fp32 bit patterns), ties to even. A non-finite input gives the IEEE result
// of the same sum (NaN as 0x7fc0).
DATTN_HD uint16_t bf16_dot2_exact(uint16_t xb, uint32_t cb, uint16_t yb, uint32_t sb) {
  const bool x_nf = (xb & 0x7f80u) == 0x7f80u, y_nf = (yb & 0x7f80u) == 0x7f80u;
  const bool c_nf = (cb & 0x7f800000u) == 0x7f800000u, s_nf = (sb & 0x7f800000u) == 0x7f800000u;
  if (x_nf || y_nf || c_nf || s_nf) {
    // infinity or NaN in a product: the sum is that of the IEEE special values
    auto special = [](uint16_t a, uint32_t b, bool a_nf, bool b_nf, int& kind, int& sign) {
      // kind: 0 finite, 1 infinite, 2 NaN
      const bool a_zero = (a & 0x7fffu) == 0, b_zero = (b & 0x7fffffffu) == 0;
      const bool a_nan = a_nf && (a & 0x7fu), b_nan = b_nf && (b & 0x7fffffu);
      sign = ((a >> 15) ^ (b >> 31)) & 1;
      if (a_nan || b_nan || (a_nf && b_zero) || (b_nf && a_zero)) kind = 2;
      else if (a_nf || b_nf) kind = 1;
      else kind = 0;
    };
    int k1, s1, k2, s2;
    special(xb, cb, x_nf, c_nf, k1, s1);
    special(yb, sb, y_nf, s_nf, k2, s2);
    if (k1 == 2 || k2 == 2 || (k1 == 1 && k2 == 1 && s1 != s2)) return 0x7fc0u;
    if (k1 == 1) return static_cast<uint16_t>(s1 ? 0xff80u : 0x7f80u);
    return static_cast<uint16_t>(s2 ? 0xff80u : 0x7f80u);
  }

  // value = (-1)^sign * m * 2^e, m an integer
  auto term = [](uint16_t a, uint32_t b, uint64_t& m, int& e, int& sign) {
    int ea = (a >> 7) & 0xff, eb = static_cast<int>((b >> 23) & 0xffu);
    uint32_t ma = a & 0x7fu, mb = b & 0x7fffffu;
    if (ea) ma |= 0x80u; else ea = 1;
    if (eb) mb |= 0x800000u; else eb = 1;
    m = static_cast<uint64_t>(ma) * mb;
    e = (ea - 134) + (eb - 150);
    sign = ((a >> 15) ^ (b >> 31)) & 1;
  };
  uint64_t mA, mB;
  int eA, eB, sA, sB;
  term(xb, cb, mA, eA, sA);
  term(yb, sb, mB, eB, sB);
  if (mA == 0 && mB == 0) return static_cast<uint16_t>((sA & sB) ? 0x8000u : 0u);

  // exact (or rounded-to-odd) signed integer V and exponent e of the sum
  int64_t V;
  int e;
  if (mA == 0 || mB == 0) {
    V = mA == 0 ? (sB ? -static_cast<int64_t>(mB) : static_cast<int64_t>(mB))
                : (sA ? -static_cast<int64_t>(mA) : static_cast<int64_t>(mA));
    e = mA == 0 ? eB : eA;
  } else {
    // normalise both significands to [2^31, 2^32) so that exponents order magnitudes
    const int nA = clz64_portable(mA) - 32, nB = clz64_portable(mB) - 32;
    mA <<= nA;
    eA -= nA;
    mB <<= nB;
    eB -= nB;
    uint64_t mH = mA, mL = mB;
    int eH = eA, eL = eB, sH = sA, sL = sB;
    if (eB > eA) {
      mH = mB; mL = mA; eH = eB; eL = eA; sH = sB; sL = sA;
    }
    const int d = eH - eL;
    if (d <= 30) {
      const int64_t h = static_cast<int64_t>(mH << d), l = static_cast<int64_t>(mL);
      V = (sH ? -h : h) + (sL ? -l : l);
      e = eL;
    } else {
      // |L| < 2^-29 |H|: keep H at 62 bits, L's bits below them become a sticky bit
      const int64_t h = static_cast<int64_t>(mH << 30);
      const int sh = d - 30;
      const uint64_t lq = sh >= 64 ? 0 : (mL >> sh);
      const bool sticky = sh >= 64 ? true : (mL & ((uint64_t{1} << sh) - 1)) != 0;
      V = (sH ? -h : h) + (sL ? -static_cast<int64_t>(lq) : static_cast<int64_t>(lq));
      e = eH - 30;
      // the exact sum lies strictly between V and V + (sL ? -1 : 1): take the odd one
      if (sticky && (V & 1) == 0) V += sL ? -1 : 1;
    }
  }
  if (V == 0) return 0;  // exact cancellation: +0

  // round |V| * 2^e to bf16: 8 significant bits, or the subnormal grid 2^-133
  const uint16_t sign = V < 0 ? 0x8000u : 0u;
  const uint64_t M = V < 0 ? static_cast<uint64_t>(-V) : static_cast<uint64_t>(V);
  const int n = 64 - clz64_portable(M);  // bit length
  const int E = e + n - 1;               // exponent of the leading bit
  int shift = E >= -126 ? n - 8 : -133 - e;
  uint64_t q;
  if (shift <= 0) {
    q = M << (-shift);
  } else if (shift >= 64) {
    q = 0;  // below half of the smallest subnormal
  } else {
    q = M >> shift;
    const uint64_t rem = M & ((uint64_t{1} << shift) - 1), half = uint64_t{1} << (shift - 1);
    if (rem > half || (rem == half && (q & 1))) ++q;
  }
  if (E < -126) return static_cast<uint16_t>(sign | q);  // subnormal (q == 128: smallest normal)
  if (q == 256) {
    q = 128;
    ++shift;
  }
  const int biased = e + shift + 7 + 127;
  if (biased >= 255) return static_cast<uint16_t>(sign | 0x7f80u);
  return static_cast<uint16_t>(sign | (biased << 7) | (q & 0x7fu));
}

// fp32 operations that the compiler may not fuse or reorder.
#if defined(__CUDA_ARCH__)
DATTN_HD float f32_mul(float a, float b) { return __fmul_rn(a, b); }
DATTN_HD float f32_add(float a, float b) { return __fadd_rn(a, b); }
DATTN_HD float f32_fma(float a, float b, float c) { return __fmaf_rn(a, b, c); }
DATTN_HD uint32_t f32_bits(float x) { return __float_as_uint(x); }
DATTN_HD float f32_of(uint32_t b) { return __uint_as_float(b); }
#else
DATTN_HD float f32_mul(float a, float b) { return a * b; }  // built without contraction
DATTN_HD float f32_add(float a, float b) { return a + b; }
DATTN_HD float f32_fma(float a, float b, float c) { return __builtin_fmaf(a, b, c); }
DATTN_HD uint32_t f32_bits(float x) { uint32_t b; __builtin_memcpy(&b, &x, 4); return b; }
DATTN_HD float f32_of(uint32_t b) { float x; __builtin_memcpy(&x, &b, 4); return x; }
#endif

// The same result as bf16_dot2_exact, mostly from fp32 arithmetic. Each product
// is split into its fp32 rounding and the exact error of that rounding (an
// FMA), the two roundings are added with the exact error of that sum
// (TwoSum), and the three error terms are added on top: the fp32 value v so
// obtained is within one unit in its last place of the exact sum, as long as
// no term is subnormal and v is not much smaller than the products (then the
// rounding errors of the error terms stay far below that unit). bf16 rounding
// only changes at the midpoints between bf16 values - fp32 patterns whose low
// 16 bits are 0x8000 - so when v is at least 3 units away from one, v and
// the exact sum round to the same bf16 value. All other cases (near a
// midpoint, cancellation, tiny or huge magnitudes, non-finite inputs) take
// the integer routine.
DATTN_HD uint16_t bf16_dot2(uint16_t xb, uint32_t cb, uint16_t yb, uint32_t sb) {
  const float x = f32_of(static_cast<uint32_t>(xb) << 16), y = f32_of(static_cast<uint32_t>(yb) << 16);
  const float c = f32_of(cb), s = f32_of(sb);
  const float ph = f32_mul(x, c), qh = f32_mul(y, s);
  const float pl = f32_fma(x, c, -ph), ql = f32_fma(y, s, -qh);
  const float sh = f32_add(ph, qh);
  // TwoSum: e1 = (ph + qh) - sh exactly
  const float bv = f32_add(sh, -ph);
  const float av = f32_add(sh, -bv);
  const float e1 = f32_add(f32_add(ph, -av), f32_add(qh, -bv));
  const float r = f32_add(f32_add(e1, pl), ql);
  const float v = f32_add(sh, r);
  const uint32_t vb = f32_bits(v);
  const uint32_t ev = (vb >> 23) & 0xffu;
  const uint32_t ep = (f32_bits(ph) >> 23) & 0xffu, eq = (f32_bits(qh) >> 23) & 0xffu;
  const uint32_t em = ep > eq ? ep : eq;  // exponent of the larger product
  const uint32_t low = vb & 0xffffu;
  // finite, normal products in [2^-60, 2^120), v within 2^-16 of the larger
  // one, and not within 2 units of a bf16 midpoint
  const bool ok = em >= 67u && em < 247u && ev + 16u >= em && ev >= 27u && (low < 0x7ffdu || low > 0x8003u);
  if (ok) return static_cast<uint16_t>((vb + 0x8000u) >> 16);
  return bf16_dot2_exact(xb, cb, yb, sb);
}

}  // namespace dattn
