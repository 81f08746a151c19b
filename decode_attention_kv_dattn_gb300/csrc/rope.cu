// RoPE prologue of a decode or verify call, and the bulk append kernel.
//
// Per-layer-type RoPE ("vllm-omni commits", Spark model commit): sliding
// layers turn all 256 head dims with theta 1e4, full layers the first quarter
// with theta 5e6. Pair i of the first r dims is (i, i + r/2) and turns by
// pos * theta^(-2i/r) (rotate-half convention); dims >= r pass through.
//
// Rounding contract of the K entry (the value stored in the cache and scored
// for the new token): c and s are the fp32 cosine and sine that rope_cos_sin
// derives from the pair's fixed-point phase step (an exact phase, then an fp32
// polynomial); the entry is the bf16 nearest to the exact x*c - y*s (ties to
// even), from fp32 error terms or, near a bf16 midpoint, in integers
// (bf16_dot2). q is rotated in fp32 and pre-scaled by log2(e)/sqrt(D) so that
// the split kernel's scores are in base-2 units; the tensor-core pass reads
// it as two bf16 terms (hi + lo, 16 significant bits), written beside it.
#include <cuda_fp16.h>

#include "bf16_exact.h"
#include "common.cuh"
#include "qk_norm.cuh"
#include "round_f64.h"

namespace dattn {

namespace {

constexpr int kRopeThreads = 64;      // append kernel
constexpr int kMaxAppendHeads = 64;   // Hkv of the append kernel
constexpr int kRowThreads = 512;      // prologue: one CTA per token row
constexpr int kMaxItems = 8;          // pair slots per thread (heads * D/2 <= 512 * 8)
constexpr int kMaxT = 16;             // verify rows per stream
constexpr int kMaxHeads = 64;         // Hq + Hkv of the prologue (heads * D/2 <= 512 * 8)

// The prologue of a call: one CTA per token row. Work items are "pair slots"
// of every head (Hq query heads, then Hkv key heads): slot p < r/2 is the
// rotated pair (p, p + r/2); slot p >= r/2 holds two pass-through dims. All
// inputs are loaded first, before waiting for the preceding launch; the
// cos/sin of each pair index is computed once per row (one thread each) into
// shared memory meanwhile. With QK-norm each head's scale comes first (one
// warp per head) and the pair slots hold the normalised bf16 values.
__global__ void __launch_bounds__(kRowThreads) rope_kernel(const RopeArgs a) {
  __shared__ float cs_c[128], cs_s[128];
  __shared__ int64_t pos_s;
  __shared__ int par_s[kMaxT];
  __shared__ double inv_s[kMaxHeads];
  // Everything up to the stores reads caller inputs only, so it runs while the
  // previous launch finishes; the workspace written below may still be read
  // by it, so the stores wait.
  const int row = blockIdx.x;
  const int half = a.r / 2;
  const int slots = a.D / 2;
  const int heads = a.Hq + a.Hkv;
  const int items = heads * slots;

  // the caller's row of this token (a prefill chunk reads a window of a
  // longer array; rows past its end read as zero)
  const int T_ = a.T > 0 ? a.T : 1;
  const int rs = row / T_, ri = row - rs * T_;
  const bool src_ok = a.row0 + ri < a.in_T;
  const int64_t src_row = static_cast<int64_t>(rs) * a.in_T + a.row0 + ri;
  auto head_src = [&](int hh) {
    return hh < a.Hq ? a.q + (src_row * a.Hq + hh) * a.D
                     : a.k + (src_row * a.Hkv + (hh - a.Hq)) * a.D;
  };
  auto head_norm = [&](int hh) { return hh < a.Hq ? a.q_norm : a.k_norm; };
  const bool norm = a.q_norm || a.k_norm;
  if (norm) {
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int hh = w; hh < heads; hh += kRowThreads / 32)
      if (head_norm(hh) && src_ok) {
        const double inv = qk_norm_inv(head_src(hh), a.D, a.norm_eps, lane);
        if (lane == 0) inv_s[hh] = inv;
      }
    __syncthreads();
  }

  // ---- loads of this thread's pair slots (independent of the position)
  uint32_t xy[kMaxItems];
#pragma unroll
  for (int k = 0; k < kMaxItems; ++k) {
    const int it = threadIdx.x + k * kRowThreads;
    xy[k] = 0;
    if (it < items && src_ok) {
      const int hh = it / slots, p = it - hh * slots;
      const uint16_t* src = head_src(hh);
      const int d0 = p < half ? p : a.r + 2 * (p - half);
      const int d1 = p < half ? p + half : d0 + 1;
      uint16_t x = src[d0], y = src[d1];
      if (norm) {
        const uint16_t* wt = head_norm(hh);
        if (wt) {
          x = qk_norm_apply(x, wt[d0], inv_s[hh]);
          y = qk_norm_apply(y, wt[d1], inv_s[hh]);
        }
      }
      xy[k] = static_cast<uint32_t>(x) | (static_cast<uint32_t>(y) << 16);
    }
  }
  // ---- position of the row
  if (a.parent) {
    const int T = a.T;
    const int s = row / T, i = row - s * T;
    if (threadIdx.x < T) par_s[threadIdx.x] = a.parent[static_cast<int64_t>(s) * T + threadIdx.x];
    __syncthreads();
    if (threadIdx.x == 0) {
      int depth = 0, node = i;
      for (int steps = 0; steps < T; ++steps) {
        const int p = par_s[node];
        if (p < 0) break;
        if (p >= node) {
          raise_error(a.err, ERR_INDEX);
          break;
        }
        ++depth;
        node = p;
      }
      pos_s = static_cast<int64_t>(a.prefix_len[s]) + depth;
    }
  } else if (threadIdx.x == 0) {
    pos_s = a.pos[row];
  }
  __syncthreads();
  if (threadIdx.x < half) {
    float cf, sf;
    rope_cos_sin(pos_s, a.rope_step[threadIdx.x], cf, sf);
    cs_c[threadIdx.x] = cf;
    cs_s[threadIdx.x] = sf;
  }
  __syncthreads();

  pdl_wait();
  pdl_trigger();

  // ---- rotate and store
#pragma unroll
  for (int k = 0; k < kMaxItems; ++k) {
    const int it = threadIdx.x + k * kRowThreads;
    if (it >= items) break;
    const int hh = it / slots, p = it - hh * slots;
    const int d0 = p < half ? p : a.r + 2 * (p - half);
    const int d1 = p < half ? p + half : d0 + 1;
    const float x = bf16_to_f32(static_cast<uint16_t>(xy[k] & 0xffffu));
    const float y = bf16_to_f32(static_cast<uint16_t>(xy[k] >> 16));
    if (hh < a.Hq) {
      const int64_t o = (static_cast<int64_t>(row) * a.Hq + hh) * a.D;
      float v0, v1;
      if (p < half) {
        const float cf = cs_c[p], sf = cs_s[p];
        v0 = fmaf(x, cf, -y * sf) * a.q_scale;
        v1 = fmaf(y, cf, x * sf) * a.q_scale;
      } else {
        v0 = x * a.q_scale;
        v1 = y * a.q_scale;
      }
      a.qhat[o + d0] = v0;
      a.qhat[o + d1] = v1;
      if (a.qhl) {
        // the tensor-core pass's operand: each value as two bf16 terms, the
        // nearest bf16 and the nearest bf16 to what is left
        const uint16_t h0 = f32_to_bf16(v0), h1 = f32_to_bf16(v1);
        const int64_t plane = static_cast<int64_t>(a.qhl_rows) * a.Hq * a.D;
        a.qhl[o + d0] = h0;
        a.qhl[o + d1] = h1;
        a.qhl[plane + o + d0] = f32_to_bf16(v0 - bf16_to_f32(h0));
        a.qhl[plane + o + d1] = f32_to_bf16(v1 - bf16_to_f32(h1));
      }
    } else {
      uint16_t* dst = a.khat + (static_cast<int64_t>(row) * a.Hkv + (hh - a.Hq)) * a.D;
      if (p < half) {
        const uint32_t cb = __float_as_uint(cs_c[p]), sb = __float_as_uint(cs_s[p]);
        const uint16_t xh = static_cast<uint16_t>(xy[k] & 0xffffu), yh = static_cast<uint16_t>(xy[k] >> 16);
        dst[d0] = bf16_dot2(xh, cb, yh, sb ^ 0x80000000u);  // x c - y s
        dst[d1] = bf16_dot2(yh, cb, xh, sb);                // y c + x s
      } else {
        dst[d0] = static_cast<uint16_t>(xy[k] & 0xffffu);
        dst[d1] = static_cast<uint16_t>(xy[k] >> 16);
      }
    }
  }
}

// One CTA per (token t, call row b): writes the token's K/V rows of every KV
// head into its ring slot or page slot.
__global__ void __launch_bounds__(kRopeThreads) append_kernel(const AppendArgs a) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x, b = blockIdx.y;
  const CacheView& c = a.c;
  const int cnt = a.count[b];
  // a ring row takes at most R tokens per call, so no slot is written twice
  if (cnt < 0 || cnt > a.Tmax || (!c.paged && cnt > c.R)) {
    if (t == 0 && threadIdx.x == 0) raise_error(a.err, ERR_INDEX);
    return;
  }
  if (t >= cnt) return;
  int src_t = t;
  if (a.gather) {
    // the row's accepted nodes must form a path from a root: else nothing of
    // the row is written
    const int32_t* acc = a.gather + static_cast<int64_t>(b) * a.Tmax;
    const int32_t* par = a.parent + static_cast<int64_t>(b) * a.in_T;
    for (int d = 0; d < cnt; ++d) {
      const int node = acc[d];
      if (node < 0 || node >= a.Tmax || par[node] != (d == 0 ? -1 : acc[d - 1])) {
        if (t == 0 && threadIdx.x == 0) raise_error(a.err, ERR_INDEX);
        return;
      }
    }
    src_t = acc[t];
  }
  const int64_t idx = static_cast<int64_t>(a.start_index[b]) + t;
  if (idx < 0) {
    if (threadIdx.x == 0) raise_error(a.err, ERR_INDEX);
    return;
  }
  // Destination row base for KV head 0; heads are D * rows_per_head apart.
  int64_t dst0;
  int64_t head_stride;
  if (c.paged) {
    const int64_t pi = idx / c.P;
    const int pg = pi < c.bt_stride ? c.block_table[static_cast<int64_t>(b) * c.bt_stride + pi] : -1;
    if (pg < 0 || pg >= c.n_rows) {
      if (threadIdx.x == 0) raise_error(a.err, ERR_INDEX);
      return;
    }
    dst0 = (static_cast<int64_t>(pg) * a.Hkv * c.P + idx % c.P) * a.D;
    head_stride = static_cast<int64_t>(c.P) * a.D;
  } else {
    const int row = c.stream_rows ? c.stream_rows[b] : b;
    if (row < 0 || row >= c.n_rows) {
      if (threadIdx.x == 0) raise_error(a.err, ERR_INDEX);
      return;
    }
    dst0 = (static_cast<int64_t>(row) * a.Hkv * c.R + idx % c.R) * a.D;
    head_stride = static_cast<int64_t>(c.R) * a.D;
  }
  const int64_t src0 = (static_cast<int64_t>(b) * a.in_T + a.row0 + src_t) * a.Hkv * a.D;
  if (a.f8) {
    // E4M3 pools (rows of D bytes): every element quantised on its own; the
    // key from its entry (QK-norm and RoPE as below when rotating)
    uint8_t* k8 = reinterpret_cast<uint8_t*>(c.k);
    uint8_t* v8 = reinterpret_cast<uint8_t*>(c.v);
    __shared__ double inv8[kMaxAppendHeads];
    const uint16_t* kn8 = a.rotate ? a.k_norm : nullptr;
    if (kn8) {
      const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
      for (int h = w; h < a.Hkv; h += kRopeThreads / 32) {
        const double inv = qk_norm_inv(a.k + src0 + h * a.D, a.D, a.norm_eps, lane);
        if (lane == 0) inv8[h] = inv;
      }
      __syncthreads();
    }
    auto kv = [&](int h, int d) {
      const uint16_t x = a.k[src0 + h * a.D + d];
      return kn8 ? qk_norm_apply(x, kn8[d], inv8[h]) : x;
    };
    const int half = a.r / 2;
    const int64_t pos = a.start_pos ? static_cast<int64_t>(a.start_pos[b]) + t : 0;
    for (int e = threadIdx.x; e < a.Hkv * a.D; e += kRopeThreads) {
      const int h = e / a.D, d = e - h * a.D;
      uint16_t entry = kv(h, d);
      if (a.rotate && d < a.r) {
        const int i = d < half ? d : d - half;
        float cf, sf;
        rope_cos_sin(pos, a.rope_step[i], cf, sf);
        const uint32_t cb = __float_as_uint(cf), sb = __float_as_uint(sf);
        entry = d < half ? bf16_dot2(kv(h, d), cb, kv(h, d + half), sb ^ 0x80000000u)  // x c - y s
                         : bf16_dot2(kv(h, d), cb, kv(h, d - half), sb);               // y c + x s
      }
      const int64_t o = dst0 + h * head_stride + d;
      k8[o] = e4m3_from_f64(static_cast<double>(bf16_to_f32(entry)) / static_cast<double>(a.k_scale));
      v8[o] = e4m3_from_f64(static_cast<double>(bf16_to_f32(a.v[src0 + h * a.D + d])) /
                            static_cast<double>(a.v_scale));
    }
    return;
  }
  // V: plain copy, 16 bytes per thread-step.  (Every return above is taken by
  // the whole CTA.)
  for (int e = threadIdx.x; e < a.Hkv * a.D / 8; e += kRopeThreads) {
    const int h = e / (a.D / 8), d8 = e % (a.D / 8);
    const uint4 w = *reinterpret_cast<const uint4*>(a.v + src0 + h * a.D + d8 * 8);
    *reinterpret_cast<uint4*>(c.v + dst0 + h * head_stride + d8 * 8) = w;
  }
  // K: the QK-norm scale of each head first (one warp per head)
  __shared__ double inv_s[kMaxAppendHeads];
  const uint16_t* kn = a.rotate ? a.k_norm : nullptr;
  if (kn) {
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int h = w; h < a.Hkv; h += kRopeThreads / 32) {
      const double inv = qk_norm_inv(a.k + src0 + h * a.D, a.D, a.norm_eps, lane);
      if (lane == 0) inv_s[h] = inv;
    }
    __syncthreads();
  }
  // one cached K value: the input, or its QK-norm
  auto kval = [&](int h, int d) {
    const uint16_t x = a.k[src0 + h * a.D + d];
    return kn ? qk_norm_apply(x, kn[d], inv_s[h]) : x;
  };
  if (!a.rotate || (a.r == 0 && !kn)) {
    for (int e = threadIdx.x; e < a.Hkv * a.D / 8; e += kRopeThreads) {
      const int h = e / (a.D / 8), d8 = e % (a.D / 8);
      const uint4 w = *reinterpret_cast<const uint4*>(a.k + src0 + h * a.D + d8 * 8);
      *reinterpret_cast<uint4*>(c.k + dst0 + h * head_stride + d8 * 8) = w;
    }
    return;
  }
  const int half = a.r / 2;
  const int64_t pos = static_cast<int64_t>(a.start_pos[b]) + t;
  for (int job = threadIdx.x; job < half + (a.D - a.r); job += kRopeThreads) {
    if (job < half) {
      const int i = job;
      float cf, sf;
      rope_cos_sin(pos, a.rope_step[i], cf, sf);
      const uint32_t cb = __float_as_uint(cf), sb = __float_as_uint(sf);
      for (int h = 0; h < a.Hkv; ++h) {
        const uint16_t x = kval(h, i), y = kval(h, i + half);
        c.k[dst0 + h * head_stride + i] = bf16_dot2(x, cb, y, sb ^ 0x80000000u);
        c.k[dst0 + h * head_stride + i + half] = bf16_dot2(y, cb, x, sb);
      }
    } else {
      const int d = a.r + (job - half);
      for (int h = 0; h < a.Hkv; ++h) c.k[dst0 + h * head_stride + d] = kval(h, d);
    }
  }
}

// The cache state, token count and root position of one prefill chunk, per
// stream (PrefillMetaArgs). A stream with metadata out of range is reported
// and gets no tokens.
__global__ void __launch_bounds__(128) prefill_meta_kernel(const PrefillMetaArgs a) {
  const CacheView& c = a.c;
  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < a.S; s += gridDim.x * blockDim.x) {
    int cnt = a.count[s];
    bool bad = cnt < 0 || cnt > a.Tmax;
    if (!c.paged) {
      const int hd = c.ring_head[s], rc = c.ring_count[s];
      bad = bad || hd < 0 || hd >= c.R || rc < 0 || rc > c.R;
      const int m = bad ? 0 : min(cnt, a.row0);
      a.head_c[s] = bad ? 0 : (hd + m) % c.R;
      a.cnt_c[s] = bad ? 0 : min(rc + m, c.R);
    } else {
      const int n = c.seq_len[s];
      bad = bad || n < 0;
      a.seq_c[s] = bad ? 0 : n + min(cnt, a.row0);
    }
    if (bad) {
      if (a.row0 == 0) raise_error(a.err, ERR_INDEX);
      cnt = 0;
    }
    a.pos_c[s] = a.start_pos ? a.start_pos[s] + a.row0 : 0;
    a.n_c[s] = max(0, min(cnt - a.row0, a.Tc));
    for (int i = 0; i < a.Tc; ++i) a.chain[s * a.Tc + i] = i - 1;
  }
}

}  // namespace

cudaError_t launch_prefill_meta(const PrefillMetaArgs& a, cudaStream_t s) {
  prefill_meta_kernel<<<(a.S + 127) / 128, 128, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rope(const RopeArgs& a, cudaStream_t s, bool pdl) {
  if ((a.Hq + a.Hkv) * (a.D / 2) > kRowThreads * kMaxItems || a.Hq + a.Hkv > kMaxHeads || a.r > 256 ||
      (a.parent && a.T > kMaxT))
    return cudaErrorNotSupported;
  if (!pdl) {  // after a launch whose outputs it reads before its wait
    rope_kernel<<<a.rows, kRowThreads, 0, s>>>(a);
    return cudaGetLastError();
  }
  return launch_pdl(rope_kernel, dim3(a.rows), dim3(kRowThreads), 0, s, a);
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
  if (a.Hkv > kMaxAppendHeads) return cudaErrorNotSupported;
  dim3 grid(a.Tmax, a.B);
  return launch_pdl(append_kernel, grid, dim3(kRopeThreads), 0, s, a);
}

}  // namespace dattn
