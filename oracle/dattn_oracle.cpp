// dattn oracle: a plain, slow fp64 CPU definition of one-token-per-stream decode
// attention over per-stream KV caches, and of tree-verify windows.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the library's product path links,
// loads or calls this file; it shares no code, header, table or constant with
// the CUDA library. Only the test suite, the smoke check and the benchmark's
// CPU-baseline leg use it.
//
// Sources (page title, passage):
//  * "vllm-omni commits" (Spark export), the score-space join commit: the cache
//    and the new token are scored separately and the two score vectors are
//    concatenated; the sliding cache is a ring of window-1 slots that needs no
//    reordering, only a mask for unwritten slots; each layer returns the new
//    K/V entry for the runtime to drop into its ring slot.
//  * same page, the Spark model commit: sliding layers rotate all 256 head dims
//    with theta 1e4, full layers the first quarter with theta 5e6; a head-wise
//    sigmoid output gate scales each head's attention output.
//  * same page, the talker export commit: grouped-query attention by reshaping
//    the query (contiguous groups of query heads share one KV head).
//  * "TensorFold PR #608": verify windows of up to 16 streams x 16 rows, each
//    row under its own tree mask; a verify row equals serial decode.
//  * "pega-omni PR #4": paged KV leases addressed through a page table.
//
// Readings where the pages are silent (each is listed in the design notes):
//  R1 RoPE pairs (i, i + r/2) inside the first r dims (rotate-half); the
//     frequencies are theta^(-2i/r); dims >= r pass through.
//  R2 score scale 1/sqrt(head_dim), no softcap.
//  R3 query head h uses KV head h / G, G = Hq / Hkv.
//  R5 a ring's valid slots are the `count` slots before `head` (cyclically);
//     the new entry is written at `head`.
//  R6 the new K entry is bf16_RNE(x*c - y*s) computed in fp64, with c and s
//     the fp32 cosine and sine of the angle pos * inv_freq given by the fixed
//     procedure in rope_cos_sin (fixed-point phase, fp32 polynomial). The
//     new token is scored with that bf16 entry, i.e. exactly the value that is
//     stored in the cache, so the score-space join equals attention over the
//     concatenated key matrix.
//  R7 gate: out = sigmoid(g_h) * attention output of head h.
//  R10 tree rows: parent[i] < i, -1 marks a root; depth(root) = 0; row i sits
//     at position prefix_len + depth(i) and attends to the prefix, its
//     ancestors and itself.
//
// Build: g++ -O2 -std=c++17 -shared -fPIC -ffp-contract=off (oracle/build.py).
// A compile-time ORACLE_MUTATION=n plants one known mistake, so the test suite
// can show that its pins catch it; the default build plants none.

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

namespace {

// ---------------------------------------------------------------- numbers

double bf16_value(uint16_t h) {
  uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// Round an fp64 value to the nearest bf16, ties to even, in one step (no
// intermediate fp32 rounding). bf16 keeps 8 significant bits and fp32's
// exponent range, so the spacing of representable values around |t| is
// 2^(e-7), with e the exponent of the leading bit, clamped at -126 below which
// the spacing is that of the subnormals.
uint16_t bf16_round(double t) {
  if (std::isnan(t)) return 0x7fc0;
  if (std::isinf(t)) return t > 0 ? 0x7f80 : 0xff80;
  if (t == 0.0) return std::signbit(t) ? 0x8000 : 0x0000;
  int e2;
  std::frexp(std::fabs(t), &e2);  // |t| = f * 2^e2, f in [0.5, 1)
  int lead = e2 - 1;
  if (lead < -126) lead = -126;
  const double spacing = std::ldexp(1.0, lead - 7);
#if ORACLE_MUTATION == 14
  double q = std::trunc(t / spacing) * spacing;  // planted: truncation
#else
  double q = std::nearbyint(t / spacing) * spacing;  // default mode: nearest-even
#endif
  if (std::fabs(q) >= std::ldexp(1.0, 128)) return std::signbit(t) ? 0xff80 : 0x7f80;
  float f = static_cast<float>(q);  // exact: q has at most 8 significant bits
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  return static_cast<uint16_t>(u >> 16);
}

// Round the exact sum p + q of two fp64 values to the nearest bf16, ties to
// even (reading R6: no intermediate rounding). hi = fl64(p + q) and the exact
// error lo (Knuth's TwoSum) give p + q = hi + lo exactly, with |lo| at most
// half an fp64 ulp of hi. A bf16 rounding tie is an fp64 value, so lo can
// only matter when hi is exactly on a tie; then it says which side p + q is.
uint16_t bf16_round_sum(double p, double q) {
  const double hi = p + q;
  if (!std::isfinite(hi) || hi == 0.0) return bf16_round(hi);
  const double bv = hi - p;
  const double lo = (p - (hi - bv)) + (q - bv);
  int e2;
  std::frexp(std::fabs(hi), &e2);
  int lead = e2 - 1;
  if (lead < -126) lead = -126;
  const double spacing = std::ldexp(1.0, lead - 7);
  const double units = hi / spacing;  // exact: a power-of-two scaling
  const double below = std::floor(units);
#if ORACLE_MUTATION == 17
  (void)below;
  return bf16_round(hi);  // planted: the fp64-rounded sum decides ties
#else
  if (lo == 0.0 || units - below != 0.5) return bf16_round(hi);
  return bf16_round((below + (lo > 0.0 ? 1.0 : 0.0)) * spacing);
#endif
}

// ---------------------------------------------------------------- RoPE (R1, R6)

// cos and sin of the rotation of pair i at position pos, as fp32 values, by
// the fixed procedure of reading R6, which the GPU runs with the same integer
// and IEEE operations:
//  1. The angle pos * theta^(-2i/r) is carried as a fraction of a turn in
//     64-bit fixed point: F = rint(2^64 * fl64(inv_freq / fl64(2 pi))), and
//     phase = pos * F mod 2^64 (exact wrap-around arithmetic; a negative pos
//     wraps the same way). Only the top 32 bits of the phase are kept.
//  2. The phase is split into a quadrant j (the turn rounded to the nearest
//     quarter) and a remainder rho in [-2^29, 2^29), i.e. [-1/8, 1/8) of a turn;
//     t = fl32(fl32(rho) * fl32(2 pi / 2^32)) is the remainder in radians.
//  3. sin t = t + t^3 (S3 + t^2 (S5 + t^2 (S7 + t^2 S9))) and
//     cos t = 1 + t^2 (C2 + t^2 (C4 + t^2 (C6 + t^2 (C8 + t^2 C10)))), in fp32
//     with fused multiply-adds, the Taylor coefficients +-1/n! rounded to fp32
//     (the first omitted terms are below 2e-9 for |t| <= pi/4).
//  4. (cos, sin) of the angle follow from (cos t, sin t) by the quarter turns j.
// The results lie within 2.5e-7 of the cosine and sine of the exact angle.
void rope_cos_sin(int r, double theta, int64_t pos, int i, double* c, double* s) {
#if ORACLE_MUTATION == 7
  (void)r;
  const double expo = -static_cast<double>(2 * i) / 256.0;  // planted: freq over 256 dims
#else
  const double expo = -static_cast<double>(2 * i) / static_cast<double>(r);
#endif
  const double inv_freq = std::pow(theta, expo);
  const uint64_t F = static_cast<uint64_t>(std::llrint(std::ldexp(inv_freq / 6.283185307179586, 64)));
  const uint64_t phase = static_cast<uint64_t>(pos) * F;  // mod 2^64
#if ORACLE_MUTATION == 16
  // planted: quadrant by truncation, remainder in [0, 1/4) turn (not centred)
  const uint32_t w = static_cast<uint32_t>(phase >> 32);
  const int quadrant = static_cast<int>(w >> 30);
  const int32_t rho = static_cast<int32_t>(w & ((1u << 30) - 1));
#else
  const uint32_t w = static_cast<uint32_t>(phase >> 32) + (1u << 29);
  const int quadrant = static_cast<int>(w >> 30);
  const int32_t rho = static_cast<int32_t>(w & ((1u << 30) - 1)) - (1 << 29);
#endif
  const float t = static_cast<float>(rho) * 1.46291807926715968e-09f;  // 2 pi / 2^32
  const float t2 = t * t;
  float sp = std::fmaf(t2, 2.75573192e-06f, -1.98412698e-04f);
  sp = std::fmaf(t2, sp, 8.33333333e-03f);
  sp = std::fmaf(t2, sp, -1.66666667e-01f);
  const float sn = std::fmaf(t * t2, sp, t);
  float cp = std::fmaf(t2, -2.75573192e-07f, 2.48015873e-05f);
  cp = std::fmaf(t2, cp, -1.38888889e-03f);
  cp = std::fmaf(t2, cp, 4.16666667e-02f);
  cp = std::fmaf(t2, cp, -5.0e-01f);
  const float cs = std::fmaf(t2, cp, 1.0f);
  float cf, sf;
  switch (quadrant) {
    case 0: cf = cs; sf = sn; break;
#if ORACLE_MUTATION == 15
    case 1: cf = sn; sf = -cs; break;  // planted: quarter turns the wrong way
    case 2: cf = -cs; sf = -sn; break;
    default: cf = -sn; sf = cs; break;
#else
    case 1: cf = -sn; sf = cs; break;
    case 2: cf = -cs; sf = -sn; break;
    default: cf = sn; sf = -cs; break;
#endif
  }
  *c = static_cast<double>(cf);
  *s = static_cast<double>(sf);
}

// Rotate the bf16 vector x (length D) at position pos. The result is fp64;
// each product of a bf16 value and an fp32 value is exact in fp64, so the only
// rounding is that of the final difference or sum.
void rope_rotate(const uint16_t* x, int D, int r, double theta, int64_t pos, double* out) {
  for (int d = 0; d < D; ++d) out[d] = bf16_value(x[d]);
  const int half = r / 2;
  for (int i = 0; i < half; ++i) {
    double c, s;
    rope_cos_sin(r, theta, pos, i, &c, &s);
#if ORACLE_MUTATION == 6
    // planted: adjacent pairs (2i, 2i+1) instead of (i, i + r/2)
    const double a = bf16_value(x[2 * i]), b = bf16_value(x[2 * i + 1]);
    out[2 * i] = a * c - b * s;
    out[2 * i + 1] = b * c + a * s;
#elif ORACLE_MUTATION == 5
    const double a = bf16_value(x[i]), b = bf16_value(x[i + half]);
    out[i] = a * c + b * s;  // planted: wrong sign
    out[i + half] = b * c - a * s;
#else
    const double a = bf16_value(x[i]), b = bf16_value(x[i + half]);
    out[i] = a * c - b * s;
    out[i + half] = b * c + a * s;
#endif
  }
}

// The K entry the layer hands back: the rotated key rounded to bf16 (R6).
// Each element is x*c - y*s or y*c + x*s with both products exact in fp64;
// their exact sum is rounded once, to the nearest bf16.
void rope_entry(const uint16_t* x, int D, int r, double theta, int64_t pos, uint16_t* entry) {
  std::vector<double> tmp(D);
  rope_rotate(x, D, r, theta, pos, tmp.data());
  for (int d = 0; d < D; ++d) entry[d] = bf16_round(tmp[d]);
  const int half = r / 2;
  for (int i = 0; i < half; ++i) {
    double c, s;
    rope_cos_sin(r, theta, pos, i, &c, &s);
    const double a = bf16_value(x[i]), b = bf16_value(x[i + half]);
    entry[i] = bf16_round_sum(a * c, -(b * s));
    entry[i + half] = bf16_round_sum(b * c, a * s);
  }
}

// ---------------------------------------------------------------- QK-norm

// Per-head RMS norm applied to q and to the new key before RoPE ("pega-omni
// PR #4", the talker kernels: RoPE with QK-norm). Reading (the pages give no
// formula): each head vector x of length D becomes
//   y_d = w_d * x_d / sqrt(mean(x^2) + eps),
// the exact value rounded once to bf16 (the layer's type), with one weight
// vector w (bf16, [D]) per layer for q and one for k; RoPE then turns y.
void qk_norm(const uint16_t* x, const uint16_t* w, int D, double eps, uint16_t* y) {
  double ss = 0.0;
  for (int d = 0; d < D; ++d) ss += bf16_value(x[d]) * bf16_value(x[d]);
#if ORACLE_MUTATION == 19
  const double inv = 1.0 / (std::sqrt(ss / D) + eps);  // planted: eps outside the root
#elif ORACLE_MUTATION == 20
  const double inv = 1.0 / std::sqrt(ss + eps);  // planted: sum instead of mean
#else
  const double inv = 1.0 / std::sqrt(ss / D + eps);
#endif
  for (int d = 0; d < D; ++d) y[d] = bf16_round(bf16_value(w[d]) * bf16_value(x[d]) * inv);
}

// The vector RoPE turns: x itself, or its QK-norm when the layer has one.
const uint16_t* normed(const uint16_t* x, const uint16_t* w, int D, double eps, std::vector<uint16_t>& buf) {
  if (!w) return x;
  buf.resize(D);
  qk_norm(x, w, D, eps, buf.data());
  return buf.data();
}

// A layer's rotation: RoPE dims and base, and its QK-norm weights (or null).
struct Rot {
  int r;
  double theta;
  const uint16_t* qn;
  const uint16_t* kn;
  double eps;
};

double sigmoid(double g) {
#if ORACLE_MUTATION == 12
  return 1.0 / (1.0 + std::exp(g));  // planted: sigmoid(-g)
#else
  return 1.0 / (1.0 + std::exp(-g));
#endif
}

double score_scale(int D) {
#if ORACLE_MUTATION == 8
  return 1.0 / static_cast<double>(D);  // planted: 1/D
#else
  return 1.0 / std::sqrt(static_cast<double>(D));
#endif
}

int kv_head_of(int h, int Hq, int Hkv) {
#if ORACLE_MUTATION == 3
  (void)Hq;
  return h % Hkv;  // planted: interleaved groups
#else
  return h / (Hq / Hkv);
#endif
}

// ---------------------------------------------------------------- attention

// One query row against a list of cached (key, value) rows plus a separately
// held set of extra rows (the new token, or a verify row's tree path), joined
// in score space: the two score vectors are concatenated, then one softmax.
//   cached_k[t], cached_v[t]: bf16 rows of length D (t < n_cached)
//   extra_k[a] (fp64, already rounded to bf16 values), extra_v[a] (bf16 rows)
void attend_score_space(const double* qhat, int D,
                        const std::vector<const uint16_t*>& cached_k,
                        const std::vector<const uint16_t*>& cached_v,
                        const std::vector<const double*>& extra_k,
                        const std::vector<const uint16_t*>& extra_v,
                        double* o) {
  const double scale = score_scale(D);
  const size_t n = cached_k.size();
  std::vector<double> s_cache(n);
  for (size_t t = 0; t < n; ++t) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qhat[d] * bf16_value(cached_k[t][d]);
    s_cache[t] = acc * scale;
  }
  const size_t ne = extra_k.size();
  std::vector<double> s_extra(ne);
  for (size_t a = 0; a < ne; ++a) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qhat[d] * extra_k[a][d];
    s_extra[a] = acc * scale;
  }
  // concatenate the score vectors: [s_cache (length n) | s_extra (length ne)]
  std::vector<double> s(s_cache);
#if ORACLE_MUTATION != 2
  s.insert(s.end(), s_extra.begin(), s_extra.end());
#endif
  double m = -INFINITY;
  for (double v : s) m = std::max(m, v);
  std::vector<double> p(s.size());
  double z = 0.0;
  for (size_t t = 0; t < s.size(); ++t) {
    p[t] = std::exp(s[t] - m);
    z += p[t];
  }
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  for (size_t t = 0; t < n; ++t) {
#if ORACLE_MUTATION == 13
    const uint16_t* vrow = cached_k[t];  // planted: values taken from keys
#else
    const uint16_t* vrow = cached_v[t];
#endif
    for (int d = 0; d < D; ++d) o[d] += p[t] * bf16_value(vrow[d]);
  }
  for (size_t a = 0; a < s.size() - n; ++a)
    for (int d = 0; d < D; ++d) o[d] += p[n + a] * bf16_value(extra_v[a][d]);
  for (int d = 0; d < D; ++d) o[d] /= z;
}

// ---------------------------------------------------------------- fp8 cache
// An fp8 KV cache ("TensorFold PR #608" names the fp8 cache and leaves it
// out; reading: OCP FP8 E4M3 values with one dequantisation scale per layer
// for K and one for V, cached value = e4m3 * scale).

// Exact value of an E4M3 byte: 1 sign, 4 exponent (bias 7), 3 mantissa bits;
// no infinities, 0x7f / 0xff are NaN; subnormals are multiples of 2^-9.
double e4m3_value(uint8_t b) {
  const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
  if (e == 15 && m == 7) return std::nan("");
  const double mag = e == 0 ? std::ldexp(static_cast<double>(m), -9) : std::ldexp(8.0 + m, e - 10);
  return sign ? -mag : mag;
}

// The E4M3 byte nearest to x (ties to even); magnitudes past 448, the largest
// finite value, saturate to 448; NaN stays NaN.
uint8_t e4m3_round(double x) {
  if (std::isnan(x)) return 0x7f;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs(x);
  if (a >= 448.0) return sign | 0x7e;
  int e2;
  std::frexp(a, &e2);                   // a = f * 2^e2, f in [0.5, 1)
  const int lead = std::max(e2 - 1, -6);  // exponent of the leading bit; subnormals share -6
  const double spacing = std::ldexp(1.0, lead - 3);
#if ORACLE_MUTATION == 24
  const double q = std::floor(a / spacing) * spacing;  // planted: truncation
#else
  const double q = std::nearbyint(a / spacing) * spacing;  // nearest, ties to even
#endif
  if (q >= 448.0) return sign | 0x7e;
  // encode q exactly
  if (q < std::ldexp(1.0, -6)) return sign | static_cast<uint8_t>(q / std::ldexp(1.0, -9));
  int e;
  const double f = std::frexp(q, &e);  // q = f * 2^e
  const int E = e - 1 + 7;
  const int M = static_cast<int>((f * 2.0 - 1.0) * 8.0);
  return sign | static_cast<uint8_t>((E << 3) | M);
}

// attend_score_space with every row given as fp64 values
void attend_score_space_f64(const double* qhat, int D, const std::vector<const double*>& cached_k,
                            const std::vector<const double*>& cached_v, const double* extra_k,
                            const double* extra_v, double* o) {
  const double scale = score_scale(D);
  const size_t n = cached_k.size();
  std::vector<double> s(n + 1);
  for (size_t t = 0; t <= n; ++t) {
    const double* k = t < n ? cached_k[t] : extra_k;
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qhat[d] * k[d];
    s[t] = acc * scale;  // [s_cache (length n) | s_new (length 1)]
  }
  double m = -INFINITY;
  for (double v : s) m = std::max(m, v);
  double z = 0.0;
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  for (size_t t = 0; t <= n; ++t) {
    const double p = std::exp(s[t] - m);
    z += p;
    const double* v = t < n ? cached_v[t] : extra_v;
    for (int d = 0; d < D; ++d) o[d] += p * v[d];
  }
  for (int d = 0; d < D; ++d) o[d] /= z;
}

// Key-space form: the keys (already rotated, as fp64 values of bf16 numbers)
// and values are stacked into explicit matrices and attended in one pass.
void attend_key_matrix(const double* qhat, int D, const std::vector<double>& K,
                       const std::vector<double>& V, size_t rows, double* o) {
  const double scale = 1.0 / std::sqrt(static_cast<double>(D));
  std::vector<double> s(rows);
  double m = -INFINITY;
  for (size_t t = 0; t < rows; ++t) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qhat[d] * K[t * D + d];
    s[t] = acc * scale;
    m = std::max(m, s[t]);
  }
  double z = 0.0;
  for (size_t t = 0; t < rows; ++t) {
    s[t] = std::exp(s[t] - m);
    z += s[t];
  }
  for (int d = 0; d < D; ++d) {
    double acc = 0.0;
    for (size_t t = 0; t < rows; ++t) acc += s[t] * V[t * D + d];
    o[d] = acc / z;
  }
}

// Run fn(item) for item in [0, n) on n_threads threads (0 = all cores).
template <class Fn>
void parallel_for(int n, int n_threads, Fn fn) {
  if (n_threads <= 0) n_threads = static_cast<int>(std::thread::hardware_concurrency());
  if (n_threads < 1) n_threads = 1;
  if (n_threads > n) n_threads = n;
  if (n_threads <= 1) {
    for (int i = 0; i < n; ++i) fn(i);
    return;
  }
  std::atomic<int> next{0};
  std::vector<std::thread> pool;
  for (int t = 0; t < n_threads; ++t)
    pool.emplace_back([&] {
      for (int i = next.fetch_add(1); i < n; i = next.fetch_add(1)) fn(i);
    });
  for (auto& th : pool) th.join();
}

struct DecodeTail {
  const uint16_t* q;      // [B, Hq, D]
  const uint16_t* k_new;  // [B, Hkv, D]
  const uint16_t* v_new;  // [B, Hkv, D]
  const uint16_t* gate;   // [B, Hq] or null
  const int32_t* pos;     // [B]
  double* out;            // [B, Hq, D]
  uint16_t* k_entry;      // [B, Hkv, D] or null
  uint16_t* v_entry;      // [B, Hkv, D] or null
};

// Shared per-(stream, KV head) step of every decode form once the list of
// valid cached rows is known: rotate, score in score space, gate, entries.
void decode_one(int b, int j, int Hq, int Hkv, int D, const Rot& rot,
                const std::vector<const uint16_t*>& ck, const std::vector<const uint16_t*>& cv,
                const DecodeTail& a) {
  const int r = rot.r;
  const double theta = rot.theta;
  const int64_t pos = a.pos[b];
  std::vector<uint16_t> kbuf, qbuf;
  const uint16_t* kn = normed(a.k_new + (static_cast<size_t>(b) * Hkv + j) * D, rot.kn, D, rot.eps, kbuf);
  const uint16_t* vn = a.v_new + (static_cast<size_t>(b) * Hkv + j) * D;
  std::vector<uint16_t> entry(D);
  rope_entry(kn, D, r, theta, pos, entry.data());
  std::vector<double> kent(D);
  for (int d = 0; d < D; ++d) kent[d] = bf16_value(entry[d]);
  if (a.k_entry) std::memcpy(a.k_entry + (static_cast<size_t>(b) * Hkv + j) * D, entry.data(), D * 2);
  if (a.v_entry) std::memcpy(a.v_entry + (static_cast<size_t>(b) * Hkv + j) * D, vn, D * 2);
  std::vector<double> qhat(D);
  for (int h = 0; h < Hq; ++h) {
    if (kv_head_of(h, Hq, Hkv) != j) continue;
    rope_rotate(normed(a.q + (static_cast<size_t>(b) * Hq + h) * D, rot.qn, D, rot.eps, qbuf), D, r, theta, pos,
                qhat.data());
    double* o = a.out + (static_cast<size_t>(b) * Hq + h) * D;
    attend_score_space(qhat.data(), D, ck, cv, {kent.data()}, {vn}, o);
#if ORACLE_MUTATION != 4
    if (a.gate) {
      const double g = sigmoid(bf16_value(a.gate[static_cast<size_t>(b) * Hq + h]));
      for (int d = 0; d < D; ++d) o[d] *= g;
    }
#endif
  }
}

bool shape_ok(int Hq, int Hkv, int D, int r) {
  return Hq > 0 && Hkv > 0 && Hq % Hkv == 0 && D > 0 && r >= 0 && r <= D && r % 2 == 0;
}

}  // namespace

extern "C" {

// ----- numbers and RoPE, exposed for the pins

uint16_t oracle_bf16_round(double t) { return bf16_round(t); }

// bf16 nearest to the exact x*c + y*s (x, y bf16 bits; c, s fp32), for the pins.
uint16_t oracle_bf16_dot2(uint16_t x, float c, uint16_t y, float s) {
  return bf16_round_sum(bf16_value(x) * static_cast<double>(c), bf16_value(y) * static_cast<double>(s));
}

// cos and sin of pair i's rotation at pos (rope_cos_sin), for the pins.
void oracle_rope_cos_sin(int r, double theta, int64_t pos, int i, double* c, double* s) {
  rope_cos_sin(r, theta, pos, i, c, s);
}

int oracle_rope_f64(const uint16_t* x, int D, int r, double theta, int64_t pos, double* out) {
  if (D <= 0 || r < 0 || r > D || r % 2) return 1;
  rope_rotate(x, D, r, theta, pos, out);
  return 0;
}

// QK-norm of one head vector (qk_norm), for the pins.
void oracle_qk_norm(const uint16_t* x, const uint16_t* w, int D, double eps, uint16_t* y) {
  qk_norm(x, w, D, eps, y);
}

int oracle_rope_bf16(const uint16_t* x, int D, int r, double theta, int64_t pos, uint16_t* out) {
  if (D <= 0 || r < 0 || r > D || r % 2) return 1;
  rope_entry(x, D, r, theta, pos, out);
  return 0;
}

// ----- decode over a ring of R slots per (row, KV head): k_ring/v_ring are
// [n_rows, Hkv, R, D] bf16. Call row b uses ring row stream_rows[b] (identity
// if null); its valid slots are the ring_count[b] slots before ring_head[b].
int oracle_decode_ring(int B, int Hq, int Hkv, int D, int r, double theta,
                       const uint16_t* k_ring, const uint16_t* v_ring, int n_rows, int R,
                       const int32_t* stream_rows, const int32_t* ring_head,
                       const int32_t* ring_count, const uint16_t* q, const uint16_t* k_new,
                       const uint16_t* v_new, const uint16_t* gate, const int32_t* pos,
                       double* out, uint16_t* k_entry, uint16_t* v_entry, int n_threads,
                       const uint16_t* q_norm, const uint16_t* k_norm, double norm_eps) {
  if (!shape_ok(Hq, Hkv, D, r) || R <= 0) return 1;
  const Rot rot{r, theta, q_norm, k_norm, norm_eps};
  for (int b = 0; b < B; ++b) {
    const int row = stream_rows ? stream_rows[b] : b;
    if (row < 0 || row >= n_rows) return 2;
    if (ring_head[b] < 0 || ring_head[b] >= R || ring_count[b] < 0 || ring_count[b] > R) return 2;
  }
  const DecodeTail tail{q, k_new, v_new, gate, pos, out, k_entry, v_entry};
  parallel_for(B * Hkv, n_threads, [&](int item) {
    const int b = item / Hkv, j = item % Hkv;
    const int row = stream_rows ? stream_rows[b] : b;
    const size_t base = (static_cast<size_t>(row) * Hkv + j) * R;
    std::vector<const uint16_t*> ck, cv;
    for (int i = 0; i < ring_count[b]; ++i) {
#if ORACLE_MUTATION == 1
      const int slot = ((ring_head[b] - i) % R + R) % R;  // planted: off by one
#else
      const int slot = ((ring_head[b] - 1 - i) % R + R) % R;
#endif
      ck.push_back(k_ring + (base + slot) * D);
      cv.push_back(v_ring + (base + slot) * D);
    }
    decode_one(b, j, Hq, Hkv, D, rot, ck, cv, tail);
  });
  return 0;
}

// ----- decode over paged leases: k_pages/v_pages are [num_pages, Hkv, P, D]
// bf16; token t of stream b lives in page block_table[b*bt_stride + t/P] at
// offset t % P; the stream holds seq_len[b] cached tokens.
int oracle_decode_paged(int B, int Hq, int Hkv, int D, int r, double theta,
                        const uint16_t* k_pages, const uint16_t* v_pages, int num_pages, int P,
                        const int32_t* block_table, int bt_stride, const int32_t* seq_len,
                        const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                        const uint16_t* gate, const int32_t* pos, double* out,
                        uint16_t* k_entry, uint16_t* v_entry, int n_threads,
                        const uint16_t* q_norm, const uint16_t* k_norm, double norm_eps) {
  if (!shape_ok(Hq, Hkv, D, r) || P <= 0) return 1;
  const Rot rot{r, theta, q_norm, k_norm, norm_eps};
  for (int b = 0; b < B; ++b) {
    if (seq_len[b] < 0 || (seq_len[b] + P - 1) / P > bt_stride) return 2;
    for (int t = 0; t < seq_len[b]; t += P) {
      const int pg = block_table[static_cast<size_t>(b) * bt_stride + t / P];
      if (pg < 0 || pg >= num_pages) return 2;
    }
  }
  const DecodeTail tail{q, k_new, v_new, gate, pos, out, k_entry, v_entry};
  parallel_for(B * Hkv, n_threads, [&](int item) {
    const int b = item / Hkv, j = item % Hkv;
    std::vector<const uint16_t*> ck, cv;
    for (int t = 0; t < seq_len[b]; ++t) {
      const int pg = block_table[static_cast<size_t>(b) * bt_stride + t / P];
#if ORACLE_MUTATION == 11
      const int off = (t + 1) % P;  // planted: offset off by one
#else
      const int off = t % P;
#endif
      const size_t row = ((static_cast<size_t>(pg) * Hkv + j) * P + off) * D;
      ck.push_back(k_pages + row);
      cv.push_back(v_pages + row);
    }
    decode_one(b, j, Hq, Hkv, D, rot, ck, cv, tail);
  });
  return 0;
}

// ----- the key-space twin over a chronological ("roll") cache: k_chrono and
// v_chrono are [B, Hkv, cap, D] bf16, oldest first, count[b] rows valid. The
// new key is rotated, rounded to its bf16 entry and appended as one more row
// of an explicit key matrix; attention runs over that matrix.
int oracle_decode_concat(int B, int Hq, int Hkv, int D, int r, double theta,
                         const uint16_t* k_chrono, const uint16_t* v_chrono, int cap,
                         const int32_t* count, const uint16_t* q, const uint16_t* k_new,
                         const uint16_t* v_new, const uint16_t* gate, const int32_t* pos,
                         double* out, int n_threads, const uint16_t* q_norm, const uint16_t* k_norm,
                         double norm_eps) {
  if (!shape_ok(Hq, Hkv, D, r)) return 1;
  for (int b = 0; b < B; ++b)
    if (count[b] < 0 || count[b] > cap) return 2;
  parallel_for(B, n_threads, [&](int b) {
    const int G = Hq / Hkv;
    for (int h = 0; h < Hq; ++h) {
      const int j = h / G;
      const size_t base = (static_cast<size_t>(b) * Hkv + j) * cap;
      const size_t rows = static_cast<size_t>(count[b]) + 1;
      std::vector<double> K(rows * D), V(rows * D);
      for (int t = 0; t < count[b]; ++t)
        for (int d = 0; d < D; ++d) {
          K[t * D + d] = bf16_value(k_chrono[(base + t) * D + d]);
          V[t * D + d] = bf16_value(v_chrono[(base + t) * D + d]);
        }
      std::vector<uint16_t> entry(D), kbuf, qbuf;
      const size_t nb = (static_cast<size_t>(b) * Hkv + j) * D;
      rope_entry(normed(k_new + nb, k_norm, D, norm_eps, kbuf), D, r, theta, pos[b], entry.data());
      for (int d = 0; d < D; ++d) {
        K[(rows - 1) * D + d] = bf16_value(entry[d]);
        V[(rows - 1) * D + d] = bf16_value(v_new[nb + d]);
      }
      std::vector<double> qhat(D);
      rope_rotate(normed(q + (static_cast<size_t>(b) * Hq + h) * D, q_norm, D, norm_eps, qbuf), D, r, theta, pos[b],
                  qhat.data());
      double* o = out + (static_cast<size_t>(b) * Hq + h) * D;
      attend_key_matrix(qhat.data(), D, K, V, rows, o);
      if (gate) {
        const double g = 1.0 / (1.0 + std::exp(-bf16_value(gate[static_cast<size_t>(b) * Hq + h])));
        for (int d = 0; d < D; ++d) o[d] *= g;
      }
    }
  });
  return 0;
}

}  // extern "C"

namespace {

// ----- tree verify: S streams x T rows. Row i of stream s sits at position
// pos0[s] + depth(i) (depth 0 for a root); it attends to the cached entries
// its layer keeps for that depth, to its ancestors in the tree and to
// itself, each window key rotated at its own position. out [S,T,Hq,D];
// k_entry [S,T,Hkv,D] receives every window key's bf16 entry.
// ("TensorFold PR #608": verify windows under tree masks; a row equals the
// plain decode of its root-to-node path.)

// One (stream, KV head) of a verify call. cached(d, ck, cv) lists the cached
// rows a row at depth d attends to.
template <typename Cached>
void verify_unit(int s, int j, int T, int Hq, int Hkv, int D, const Rot& rot, int64_t pos0,
                 const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* parent,
                 const uint16_t* gate, double* out, uint16_t* k_entry, Cached cached) {
  const int32_t* par = parent + static_cast<size_t>(s) * T;
  // depth of each node by walking to its root
  std::vector<int> depth(T);
  for (int i = 0; i < T; ++i) {
    int dpt = 0;
    for (int a = par[i]; a >= 0; a = par[a]) ++dpt;
#if ORACLE_MUTATION == 9
    depth[i] = dpt + 1;  // planted: depth counted from 1
#else
    depth[i] = dpt;
#endif
  }
  // rotated bf16 entries of the window keys, each at its own position
  std::vector<uint16_t> ent(static_cast<size_t>(T) * D);
  std::vector<double> entd(static_cast<size_t>(T) * D);
  for (int i = 0; i < T; ++i) {
    const size_t src = ((static_cast<size_t>(s) * T + i) * Hkv + j) * D;
    std::vector<uint16_t> kbuf;
    rope_entry(normed(k + src, rot.kn, D, rot.eps, kbuf), D, rot.r, rot.theta, pos0 + depth[i],
               ent.data() + static_cast<size_t>(i) * D);
    for (int d = 0; d < D; ++d) entd[static_cast<size_t>(i) * D + d] = bf16_value(ent[static_cast<size_t>(i) * D + d]);
    if (k_entry) std::memcpy(k_entry + src, ent.data() + static_cast<size_t>(i) * D, D * 2);
  }
  std::vector<double> qhat(D);
  for (int i = 0; i < T; ++i) {
    std::vector<const uint16_t*> ck, cv;
    cached(depth[i], ck, cv);
    // the row's tree path: itself and its ancestors
    std::vector<const double*> ek;
    std::vector<const uint16_t*> ev;
#if ORACLE_MUTATION == 10
    for (int a = 0; a < T; ++a) {  // planted: no tree mask
#else
    for (int a = i; a >= 0; a = par[a]) {
#endif
      ek.push_back(entd.data() + static_cast<size_t>(a) * D);
      ev.push_back(v + ((static_cast<size_t>(s) * T + a) * Hkv + j) * D);
    }
    for (int h = 0; h < Hq; ++h) {
      if (kv_head_of(h, Hq, Hkv) != j) continue;
      const size_t qi = (static_cast<size_t>(s) * T + i) * Hq + h;
      std::vector<uint16_t> qbuf;
      rope_rotate(normed(q + qi * D, rot.qn, D, rot.eps, qbuf), D, rot.r, rot.theta, pos0 + depth[i],
                  qhat.data());
      double* o = out + qi * D;
      attend_score_space(qhat.data(), D, ck, cv, ek, ev, o);
      if (gate) {
        const double g = sigmoid(bf16_value(gate[qi]));
        for (int d = 0; d < D; ++d) o[d] *= g;
      }
    }
  }
}

bool parents_ok(int S, int T, const int32_t* parent) {
  for (int s = 0; s < S; ++s)
    for (int i = 0; i < T; ++i) {
      const int pa = parent[static_cast<size_t>(s) * T + i];
      if (pa < -1 || pa >= i) return false;
    }
  return true;
}

}  // namespace

extern "C" {

// Paged layer: a row at any depth attends to the stream's whole prefix of
// prefix_len[s] tokens; the window's root sits at pos[s], or at prefix_len[s]
// when pos is null.
int oracle_verify(int S, int T, int Hq, int Hkv, int D, int r, double theta,
                  const uint16_t* k_pages, const uint16_t* v_pages, int num_pages, int P,
                  const int32_t* block_table, int bt_stride, const int32_t* prefix_len,
                  const int32_t* pos, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                  const int32_t* parent, const uint16_t* gate, double* out,
                  uint16_t* k_entry, int n_threads, const uint16_t* q_norm, const uint16_t* k_norm,
                  double norm_eps) {
  if (!shape_ok(Hq, Hkv, D, r) || P <= 0 || T <= 0) return 1;
  for (int s = 0; s < S; ++s) {
    if (prefix_len[s] < 0 || (prefix_len[s] + P - 1) / P > bt_stride) return 2;
    for (int t = 0; t < prefix_len[s]; t += P) {
      const int pg = block_table[static_cast<size_t>(s) * bt_stride + t / P];
      if (pg < 0 || pg >= num_pages) return 2;
    }
  }
  if (!parents_ok(S, T, parent)) return 3;
  const Rot rot{r, theta, q_norm, k_norm, norm_eps};
  parallel_for(S * Hkv, n_threads, [&](int item) {
    const int s = item / Hkv, j = item % Hkv;
    std::vector<const uint16_t*> pk, pv;
    for (int t = 0; t < prefix_len[s]; ++t) {
      const int pg = block_table[static_cast<size_t>(s) * bt_stride + t / P];
      const size_t row = ((static_cast<size_t>(pg) * Hkv + j) * P + t % P) * D;
      pk.push_back(k_pages + row);
      pv.push_back(v_pages + row);
    }
    const int64_t pos0 = pos ? pos[s] : prefix_len[s];
    verify_unit(s, j, T, Hq, Hkv, D, rot, pos0, q, k, v, parent, gate, out, k_entry,
                [&](int, std::vector<const uint16_t*>& ck, std::vector<const uint16_t*>& cv) {
                  ck = pk;
                  cv = pv;
                });
  });
  return 0;
}

// Ring (sliding-window) layer: ring row stream_rows[s] (identity if null)
// holds ring_count[s] valid entries, the slots before ring_head[s]. A row at
// depth d attends to the newest min(count, R - d) of them: what the ring
// holds after its d ancestors were appended, the window keeping R cached
// tokens - the entries the plain decode of its path would see.
int oracle_verify_ring(int S, int T, int Hq, int Hkv, int D, int r, double theta,
                       const uint16_t* k_ring, const uint16_t* v_ring, int n_rows, int R,
                       const int32_t* stream_rows, const int32_t* ring_head, const int32_t* ring_count,
                       const int32_t* pos, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const int32_t* parent, const uint16_t* gate, double* out, uint16_t* k_entry,
                       int n_threads, const uint16_t* q_norm, const uint16_t* k_norm, double norm_eps) {
  if (!shape_ok(Hq, Hkv, D, r) || R <= 0 || T <= 0) return 1;
  for (int s = 0; s < S; ++s) {
    const int row = stream_rows ? stream_rows[s] : s;
    if (row < 0 || row >= n_rows) return 2;
    if (ring_head[s] < 0 || ring_head[s] >= R || ring_count[s] < 0 || ring_count[s] > R) return 2;
  }
  if (!parents_ok(S, T, parent)) return 3;
  const Rot rot{r, theta, q_norm, k_norm, norm_eps};
  parallel_for(S * Hkv, n_threads, [&](int item) {
    const int s = item / Hkv, j = item % Hkv;
    const int row = stream_rows ? stream_rows[s] : s;
    const size_t base = (static_cast<size_t>(row) * Hkv + j) * R;
    verify_unit(s, j, T, Hq, Hkv, D, rot, pos[s], q, k, v, parent, gate, out, k_entry,
                [&](int d, std::vector<const uint16_t*>& ck, std::vector<const uint16_t*>& cv) {
#if ORACLE_MUTATION == 21
                  const int keep = ring_count[s];  // planted: the path's entries drop nothing
                  (void)d;
#else
                  const int keep = std::min(ring_count[s], std::max(0, R - d));
#endif
                  ck.clear();
                  cv.clear();
                  for (int i = 0; i < keep; ++i) {  // newest first
                    const int slot = ((ring_head[s] - 1 - i) % R + R) % R;
                    ck.push_back(k_ring + (base + slot) * D);
                    cv.push_back(v_ring + (base + slot) * D);
                  }
                });
  });
  return 0;
}

// ----- bulk append. Token t (< count[b]) of call row b goes to cache index
// start_index[b] + t and, when rotate != 0, is rotated at position
// start_pos[b] + t. k/v are [B, Tmax, Hkv, D]. The caches are updated in place.
// Ring: index i of row stream_rows[b] is slot i mod R of [n_rows, Hkv, R, D];
// a call writes at most R tokens per ring row.
int oracle_append_ring(int B, int Tmax, int Hkv, int D, int r, double theta,
                       uint16_t* k_ring, uint16_t* v_ring, int n_rows, int R,
                       const int32_t* stream_rows, const int32_t* start_index,
                       const int32_t* start_pos, const int32_t* count,
                       const uint16_t* k, const uint16_t* v, int rotate, const uint16_t* k_norm,
                       double norm_eps) {
  if (D <= 0 || r < 0 || r > D || r % 2 || R <= 0) return 1;
  std::vector<uint16_t> entry(D), kbuf;
  for (int b = 0; b < B; ++b) {
    const int row = stream_rows ? stream_rows[b] : b;
    // at most one ring's worth per call: each slot is written at most once
    if (row < 0 || row >= n_rows || count[b] < 0 || count[b] > Tmax || count[b] > R || start_index[b] < 0)
      return 2;
    for (int t = 0; t < count[b]; ++t)
      for (int j = 0; j < Hkv; ++j) {
        const size_t src = ((static_cast<size_t>(b) * Tmax + t) * Hkv + j) * D;
#if ORACLE_MUTATION == 18
        const int slot = (start_index[b] + t + 1) % R;  // planted: slot off by one
#else
        const int slot = (start_index[b] + t) % R;
#endif
        const size_t dst = ((static_cast<size_t>(row) * Hkv + j) * R + slot) * D;
        if (rotate)
          rope_entry(normed(k + src, k_norm, D, norm_eps, kbuf), D, r, theta, start_pos[b] + t, entry.data());
        else
          std::memcpy(entry.data(), k + src, D * 2);
        std::memcpy(k_ring + dst, entry.data(), D * 2);
        std::memcpy(v_ring + dst, v + src, D * 2);
      }
  }
  return 0;
}

// Paged: index i of row b is offset i % P of page block_table[b*bt_stride + i/P].
int oracle_append_paged(int B, int Tmax, int Hkv, int D, int r, double theta,
                        uint16_t* k_pages, uint16_t* v_pages, int num_pages, int P,
                        const int32_t* block_table, int bt_stride, const int32_t* start_index,
                        const int32_t* start_pos, const int32_t* count,
                        const uint16_t* k, const uint16_t* v, int rotate, const uint16_t* k_norm,
                        double norm_eps) {
  if (D <= 0 || r < 0 || r > D || r % 2 || P <= 0) return 1;
  std::vector<uint16_t> entry(D), kbuf;
  for (int b = 0; b < B; ++b) {
    if (count[b] < 0 || count[b] > Tmax || start_index[b] < 0) return 2;
    if (count[b] > 0 && (start_index[b] + count[b] - 1) / P >= bt_stride) return 2;
    for (int t = 0; t < count[b]; ++t) {
      const int idx = start_index[b] + t;
      const int pg = block_table[static_cast<size_t>(b) * bt_stride + idx / P];
      if (pg < 0 || pg >= num_pages) return 2;
      for (int j = 0; j < Hkv; ++j) {
        const size_t src = ((static_cast<size_t>(b) * Tmax + t) * Hkv + j) * D;
        const size_t dst = ((static_cast<size_t>(pg) * Hkv + j) * P + idx % P) * D;
        if (rotate)
          rope_entry(normed(k + src, k_norm, D, norm_eps, kbuf), D, r, theta, start_pos[b] + t, entry.data());
        else
          std::memcpy(entry.data(), k + src, D * 2);
        std::memcpy(k_pages + dst, entry.data(), D * 2);
        std::memcpy(v_pages + dst, v + src, D * 2);
      }
    }
  }
  return 0;
}

// ----- commit of the accepted verify paths ("TensorFold PR #608": a verify
// round commits only each stream's accepted path). accepted [S, T] lists the
// accepted nodes of stream s root first, num_accepted[s] of them; they must
// form a path from a root (accepted[0] a root, each next node a child of the
// one before). Node accepted[s][d] goes to cache index start + d - ring: slot
// (ring_head[s] + d) mod R of ring row stream_rows[s]; paged: token
// seq_len[s] + d - with its key rotated at pos[s] + d: the entry that the
// verify row of that node and the plain decode of its path use. k, v are the
// verify call's window inputs [S, T, Hkv, D]. A stream whose list is not such
// a path is left unchanged, and the call then returns 3.
}  // extern "C"

namespace {
bool path_ok(int T, const int32_t* par, const int32_t* acc, int n) {
  if (n < 0 || n > T) return false;
  for (int d = 0; d < n; ++d) {
    const int a = acc[d];
    if (a < 0 || a >= T || par[a] != (d == 0 ? -1 : acc[d - 1])) return false;
  }
  return true;
}

// the accepted nodes' k and v rows gathered into [S, T, Hkv, D]; counts[s] =
// the path length, or 0 for a stream whose list is not a path
bool gather_paths(int S, int T, int Hkv, int D, const uint16_t* k, const uint16_t* v,
                  const int32_t* parent, const int32_t* accepted, const int32_t* num_accepted,
                  std::vector<uint16_t>& kg, std::vector<uint16_t>& vg, std::vector<int32_t>& counts) {
  const size_t row = static_cast<size_t>(Hkv) * D;
  kg.assign(static_cast<size_t>(S) * T * row, 0);
  vg.assign(kg.size(), 0);
  counts.assign(S, 0);
  bool all_ok = true;
  for (int s = 0; s < S; ++s) {
    const int32_t* acc = accepted + static_cast<size_t>(s) * T;
    if (!path_ok(T, parent + static_cast<size_t>(s) * T, acc, num_accepted[s])) {
      all_ok = false;
      continue;
    }
    counts[s] = num_accepted[s];
    for (int d = 0; d < counts[s]; ++d) {
#if ORACLE_MUTATION == 22
      const size_t src = (static_cast<size_t>(s) * T + d) * row;  // planted: the first nodes, not the path's
#else
      const size_t src = (static_cast<size_t>(s) * T + acc[d]) * row;
#endif
      const size_t dst = (static_cast<size_t>(s) * T + d) * row;
      std::memcpy(&kg[dst], k + src, row * 2);
      std::memcpy(&vg[dst], v + src, row * 2);
    }
  }
  return all_ok;
}
}  // namespace

extern "C" {

int oracle_commit_ring(int S, int T, int Hkv, int D, int r, double theta, uint16_t* k_ring,
                       uint16_t* v_ring, int n_rows, int R, const int32_t* stream_rows,
                       const int32_t* ring_head, const int32_t* pos, const uint16_t* k,
                       const uint16_t* v, const int32_t* parent, const int32_t* accepted,
                       const int32_t* num_accepted, const uint16_t* k_norm, double norm_eps) {
  std::vector<uint16_t> kg, vg;
  std::vector<int32_t> counts;
  const bool ok = gather_paths(S, T, Hkv, D, k, v, parent, accepted, num_accepted, kg, vg, counts);
  const int rc = oracle_append_ring(S, T, Hkv, D, r, theta, k_ring, v_ring, n_rows, R, stream_rows, ring_head,
                                    pos, counts.data(), kg.data(), vg.data(), 1, k_norm, norm_eps);
  return rc != 0 ? rc : (ok ? 0 : 3);
}

int oracle_commit_paged(int S, int T, int Hkv, int D, int r, double theta, uint16_t* k_pages,
                        uint16_t* v_pages, int num_pages, int P, const int32_t* block_table,
                        int bt_stride, const int32_t* seq_len, const int32_t* pos,
                        const uint16_t* k, const uint16_t* v, const int32_t* parent,
                        const int32_t* accepted, const int32_t* num_accepted,
                        const uint16_t* k_norm, double norm_eps) {
  std::vector<uint16_t> kg, vg;
  std::vector<int32_t> counts;
  const bool ok = gather_paths(S, T, Hkv, D, k, v, parent, accepted, num_accepted, kg, vg, counts);
  const int rc = oracle_append_paged(S, T, Hkv, D, r, theta, k_pages, v_pages, num_pages, P, block_table,
                                     bt_stride, seq_len, pos, counts.data(), kg.data(), vg.data(), 1, k_norm,
                                     norm_eps);
  return rc != 0 ? rc : (ok ? 0 : 3);
}

// ----- ragged prefill: stream s brings count[s] new tokens (q [S, Tmax, Hq, D],
// k, v [S, Tmax, Hkv, D], gate [S, Tmax, Hq] or null), token t at position
// start_pos[s] + t. Read as the plain definition: the tokens are decoded one
// after another, each one joined to the cache in score space and its entry
// written back before the next (ring: slot head + t, the ring keeping its
// newest R entries; paged: token index seq_len[s] + t), so token t attends to
// the cache and to new tokens 0..t. out [S, Tmax, Hq, D] gets rows t <
// count[s]; the caches are updated in place.
int oracle_prefill_ring(int S, int Tmax, int Hq, int Hkv, int D, int r, double theta, uint16_t* k_ring,
                        uint16_t* v_ring, int n_rows, int R, const int32_t* stream_rows, const int32_t* ring_head,
                        const int32_t* ring_count, const int32_t* count, const int32_t* start_pos,
                        const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* gate, double* out,
                        const uint16_t* q_norm, const uint16_t* k_norm, double norm_eps) {
  for (int s = 0; s < S; ++s)
    if (count[s] < 0 || count[s] > Tmax) return 2;
  const size_t qrow = static_cast<size_t>(Hq) * D, kvrow = static_cast<size_t>(Hkv) * D;
  std::vector<uint16_t> ke(kvrow), ve(kvrow);
  for (int s = 0; s < S; ++s) {
    const int row = stream_rows ? stream_rows[s] : s;
    int head = ring_head[s], cnt = ring_count[s];
    for (int t = 0; t < count[s]; ++t) {
      const size_t tok = static_cast<size_t>(s) * Tmax + t;
#if ORACLE_MUTATION == 23
      const int32_t pos = start_pos[s] + t + 1;  // planted: positions shifted by one
#else
      const int32_t pos = start_pos[s] + t;
#endif
      const int rc = oracle_decode_ring(1, Hq, Hkv, D, r, theta, k_ring, v_ring, n_rows, R, &row, &head, &cnt,
                                        q + tok * qrow, k + tok * kvrow, v + tok * kvrow,
                                        gate ? gate + tok * Hq : nullptr, &pos, out + tok * qrow, ke.data(),
                                        ve.data(), 1, q_norm, k_norm, norm_eps);
      if (rc != 0) return rc;
      for (int j = 0; j < Hkv; ++j) {
        const size_t dst = ((static_cast<size_t>(row) * Hkv + j) * R + head) * D;
        std::memcpy(k_ring + dst, ke.data() + static_cast<size_t>(j) * D, D * 2);
        std::memcpy(v_ring + dst, ve.data() + static_cast<size_t>(j) * D, D * 2);
      }
      head = (head + 1) % R;
      cnt = std::min(cnt + 1, R);
    }
  }
  return 0;
}

int oracle_prefill_paged(int S, int Tmax, int Hq, int Hkv, int D, int r, double theta, uint16_t* k_pages,
                         uint16_t* v_pages, int num_pages, int P, const int32_t* block_table, int bt_stride,
                         const int32_t* seq_len, const int32_t* count, const int32_t* start_pos,
                         const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* gate,
                         double* out, const uint16_t* q_norm, const uint16_t* k_norm, double norm_eps) {
  for (int s = 0; s < S; ++s)
    if (count[s] < 0 || count[s] > Tmax) return 2;
  const size_t qrow = static_cast<size_t>(Hq) * D, kvrow = static_cast<size_t>(Hkv) * D;
  std::vector<uint16_t> ke(kvrow), ve(kvrow);
  for (int s = 0; s < S; ++s) {
    const int32_t* bt = block_table + static_cast<size_t>(s) * bt_stride;
    for (int t = 0; t < count[s]; ++t) {
      const size_t tok = static_cast<size_t>(s) * Tmax + t;
      const int32_t pos = start_pos[s] + t, n = seq_len[s] + t;
      const int idx = n / P;
      if (idx >= bt_stride || bt[idx] < 0 || bt[idx] >= num_pages) return 2;
      const int rc = oracle_decode_paged(1, Hq, Hkv, D, r, theta, k_pages, v_pages, num_pages, P, bt, bt_stride,
                                         &n, q + tok * qrow, k + tok * kvrow, v + tok * kvrow,
                                         gate ? gate + tok * Hq : nullptr, &pos, out + tok * qrow, ke.data(),
                                         ve.data(), 1, q_norm, k_norm, norm_eps);
      if (rc != 0) return rc;
      for (int j = 0; j < Hkv; ++j) {
        const size_t dst = ((static_cast<size_t>(bt[idx]) * Hkv + j) * P + n % P) * D;
        std::memcpy(k_pages + dst, ke.data() + static_cast<size_t>(j) * D, D * 2);
        std::memcpy(v_pages + dst, ve.data() + static_cast<size_t>(j) * D, D * 2);
      }
    }
  }
  return 0;
}

// ----- E4M3 conversions, for the pins
double oracle_e4m3_value(uint8_t b) { return e4m3_value(b); }
uint8_t oracle_e4m3_round(double x) { return e4m3_round(x); }

// ----- decode over an fp8 (E4M3) cache, ring (paged == 0: k/v [n_rows, Hkv,
// R, D], valid slots the ring_count[b] before ring_head[b], stream_rows) or
// paged (k/v [n_rows pages, Hkv, P, D], block_table, seq_len). Cached K value =
// e4m3 * k_scale, V value = e4m3 * v_scale. The new token's K entry (the bf16
// nearest its exact rotation, as in the bf16 cache) and its v_new are stored
// as the E4M3 bytes nearest entry / k_scale and v_new / v_scale (fp64
// quotients), and the new token is joined in score space as stored: the
// values a later decode reads. k_entry, v_entry [B, Hkv, D] receive the bytes.
int oracle_decode_fp8(int paged, int B, int Hq, int Hkv, int D, int r, double theta, const uint8_t* k_cache,
                      const uint8_t* v_cache, int n_rows, int R_or_P, const int32_t* stream_rows,
                      const int32_t* ring_head, const int32_t* ring_count, const int32_t* block_table,
                      int bt_stride, const int32_t* seq_len, double k_scale, double v_scale, const uint16_t* q,
                      const uint16_t* k_new, const uint16_t* v_new, const uint16_t* gate, const int32_t* pos,
                      double* out, uint8_t* k_entry, uint8_t* v_entry, const uint16_t* q_norm,
                      const uint16_t* k_norm, double norm_eps) {
  if (!shape_ok(Hq, Hkv, D, r) || R_or_P <= 0 || !(k_scale > 0.0) || !(v_scale > 0.0)) return 1;
  const Rot rot{r, theta, q_norm, k_norm, norm_eps};
  for (int b = 0; b < B; ++b) {
    for (int j = 0; j < Hkv; ++j) {
      // the valid cached rows, dequantised
      std::vector<std::vector<double>> kd, vd;
      auto add = [&](size_t row) {
        kd.emplace_back(D);
        vd.emplace_back(D);
        for (int d = 0; d < D; ++d) {
#if ORACLE_MUTATION == 25
          kd.back()[d] = e4m3_value(k_cache[row * D + d]);  // planted: K scale dropped
#else
          kd.back()[d] = e4m3_value(k_cache[row * D + d]) * k_scale;
#endif
          vd.back()[d] = e4m3_value(v_cache[row * D + d]) * v_scale;
        }
      };
      if (!paged) {
        const int R = R_or_P, row = stream_rows ? stream_rows[b] : b;
        if (row < 0 || row >= n_rows || ring_head[b] < 0 || ring_head[b] >= R || ring_count[b] < 0 ||
            ring_count[b] > R)
          return 2;
        for (int i = 0; i < ring_count[b]; ++i)
          add((static_cast<size_t>(row) * Hkv + j) * R + ((ring_head[b] - 1 - i) % R + R) % R);
      } else {
        const int P = R_or_P;
        if (seq_len[b] < 0 || (seq_len[b] + P - 1) / P > bt_stride) return 2;
        for (int t = 0; t < seq_len[b]; ++t) {
          const int pg = block_table[static_cast<size_t>(b) * bt_stride + t / P];
          if (pg < 0 || pg >= n_rows) return 2;
          add((static_cast<size_t>(pg) * Hkv + j) * P + t % P);
        }
      }
      std::vector<const double*> ck, cv;
      for (size_t t = 0; t < kd.size(); ++t) {
        ck.push_back(kd[t].data());
        cv.push_back(vd[t].data());
      }
      // the new token, quantised as stored
      std::vector<uint16_t> kbuf, qbuf, entry(D);
      const size_t nb = (static_cast<size_t>(b) * Hkv + j) * D;
      rope_entry(normed(k_new + nb, rot.kn, D, rot.eps, kbuf), D, r, theta, pos[b], entry.data());
      std::vector<double> kn(D), vn(D);
      for (int d = 0; d < D; ++d) {
        const uint8_t k8 = e4m3_round(bf16_value(entry[d]) / k_scale);
        const uint8_t v8 = e4m3_round(bf16_value(v_new[nb + d]) / v_scale);
        if (k_entry) k_entry[nb + d] = k8;
        if (v_entry) v_entry[nb + d] = v8;
        kn[d] = e4m3_value(k8) * k_scale;
        vn[d] = e4m3_value(v8) * v_scale;
      }
      std::vector<double> qhat(D);
      for (int h = 0; h < Hq; ++h) {
        if (kv_head_of(h, Hq, Hkv) != j) continue;
        rope_rotate(normed(q + (static_cast<size_t>(b) * Hq + h) * D, rot.qn, D, rot.eps, qbuf), D, r, theta,
                    pos[b], qhat.data());
        double* o = out + (static_cast<size_t>(b) * Hq + h) * D;
        attend_score_space_f64(qhat.data(), D, ck, cv, kn.data(), vn.data(), o);
        if (gate) {
          const double g = sigmoid(bf16_value(gate[static_cast<size_t>(b) * Hq + h]));
          for (int d = 0; d < D; ++d) o[d] *= g;
        }
      }
    }
  }
  return 0;
}

int oracle_hardware_threads(void) {
  return static_cast<int>(std::thread::hardware_concurrency());
}

int oracle_mutation(void) { return ORACLE_MUTATION; }

}  // extern "C"
