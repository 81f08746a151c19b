// Decode attention: split-K pass over the cached keys and the LSE combine that
// joins the new token in score space.
//
// Method ("vllm-omni commits", score-space join commit): the cached keys (n of
// them) and the new key are scored separately and their score vectors meet in
// one softmax; nothing cache-sized is copied, and the new K/V entry is written
// into its slot afterwards. A ring's slots need no reordering (softmax is
// order-free, cached keys carry their own rotary phase); unwritten slots are
// masked by never being read. Grouped-query attention shares each KV head's
// loads among its G query heads ("vllm-omni commits", talker export commit).
// Splitting the keys over many CTAs and merging their partial softmax states
// follows "TensorFold PR #608" (the split "shared" kernel plus a merge, and the
// lesson that a merge must not be a chain of dependent loads).
//
// GB300 design. The KV stream is HBM-bound at G flops per byte, so the scores
// and the value sum run on the FP32 pipes, not on tensor cores. Each warp owns
// a private pipeline of KT-key tiles: one lane issues bulk TMA copies
// (cp.async.bulk, global -> shared, completion counted on an mbarrier) for K
// and V of the tile kStages ahead. A lane holds 8 dims (one 16-byte load) of a
// key; the G per-head dot products of J keys (J * G = lanes per key) are
// reduced across lanes by a transposing butterfly, which leaves exactly one
// (key, head) score per lane, so the online softmax costs one exp2 per lane per
// tile. Probabilities go through shared memory to all lanes for the value sum.
#include "common.cuh"

namespace dattn {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = 4;

template <int D, int GP>
struct Geo {
  static constexpr int LPK = D / 8;         // lanes per key row (16 bytes each)
  static constexpr int KPS = 32 / LPK;      // keys per warp-wide load
  static constexpr int J = LPK / GP;        // loads per tile (J * GP scores per lane)
  static constexpr int KT = J * KPS;        // keys per tile
  static constexpr int ROW = D * 2;         // bytes per key row
  static constexpr int TILE = KT * ROW;     // bytes of one K (or V) tile
  static constexpr int STAGE = 2 * TILE;
  // stages per warp: about 24 KB of K/V in flight per warp, at least 2
  static constexpr int NS = (24576 / STAGE) < 2 ? 2 : ((24576 / STAGE) > 8 ? 8 : 24576 / STAGE);
  static constexpr int STAGE_BYTES = kWarps * NS * STAGE;
  static constexpr int MERGE_BYTES = kWarps * GP * (D + 2) * 4;
  static constexpr int BAR_OFF = STAGE_BYTES > MERGE_BYTES ? STAGE_BYTES : MERGE_BYTES;
  static constexpr int PSM_OFF = BAR_OFF + kWarps * NS * 8;
  static constexpr int SMEM = PSM_OFF + kWarps * (32 + GP) * 4;
  static_assert(D == 128 || D == 256, "head_dim");
  static_assert(LPK % GP == 0, "GP must divide the lanes per key");
};

__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
  f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x);
  f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
  f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z);
  f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
}

// Sum N = W partial values across W lanes (W a power of two, groups aligned)
// so that lane l ends with the full sum of value (l % W). Each level halves the
// values a lane keeps: the lane whose bit `w` is set keeps the upper half and
// sends the lower half to its partner, and the other way round.
template <int W>
__device__ __forceinline__ float transpose_reduce(float (&v)[W], int lane) {
#pragma unroll
  for (int w = W / 2; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float lo = v[i], hi = v[i + w];
      const float send = upper ? lo : hi;
      const float keep = upper ? hi : lo;
      v[i] = keep + __shfl_xor_sync(kFull, send, w);
    }
  }
  return v[0];
}

// The cached keys of call row b for KV head j: count n, ring start slot and
// base pointers. Bad metadata reads nothing and is reported once.
struct StreamKeys {
  int n;
  int start;
  const uint16_t* kb;
  const uint16_t* vb;
};

template <bool PAGED, int D>
__device__ __forceinline__ StreamKeys stream_keys(const CacheView& c, int b, int j, int Hkv,
                                                  int max_len, bool report, int* err) {
  StreamKeys s{0, 0, c.k, c.v};
  if constexpr (PAGED) {
    int n = c.seq_len[b];
    const int cap = min(max_len, c.bt_stride * c.P);
    if (n < 0 || n > cap) {
      if (report) raise_error(err, ERR_LENGTH);
      n = n < 0 ? 0 : cap;
    }
    s.n = n;
  } else {
    const int row = c.stream_rows ? c.stream_rows[b] : b;
    const int head = c.ring_head[b], cnt = c.ring_count[b];
    if (row < 0 || row >= c.n_rows || head < 0 || head >= c.R || cnt < 0 || cnt > c.R) {
      if (report) raise_error(err, ERR_INDEX);
      return s;
    }
    s.n = cnt;
    s.start = head - cnt < 0 ? head - cnt + c.R : head - cnt;
    const int64_t off = (static_cast<int64_t>(row) * Hkv + j) * c.R * D;
    s.kb = c.k + off;
    s.vb = c.v + off;
  }
  return s;
}

template <int D, int GP, bool PAGED>
__global__ void __launch_bounds__(kWarps * 32, 2) decode_split_kernel(const SplitArgs a, int G) {
  using Gm = Geo<D, GP>;
  constexpr int LPK = Gm::LPK, KPS = Gm::KPS, J = Gm::J, KT = Gm::KT, NS = Gm::NS;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int split = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const CacheView& c = a.c;
  const int Hkv = a.Hkv;

  // Caller metadata and the cache itself are not written by the preceding
  // kernel (the RoPE prologue), so the first tiles are requested before the
  // dependency wait and overlap it.
  const StreamKeys sk = stream_keys<PAGED, D>(c, b, j, Hkv, a.max_len,
                                              split == 0 && threadIdx.x == 0, a.err);
  const int k0 = split * a.chunk;
  const int k1 = min(sk.n, k0 + a.chunk);
  const int ntiles = k1 > k0 ? (k1 - k0 + KT - 1) / KT : 0;
  const int my_tiles = ntiles > warp ? (ntiles - warp + kWarps - 1) / kWarps : 0;

  uint8_t* wsm = smem + warp * NS * Gm::STAGE;
  const uint32_t bar0 = smem_addr(smem + Gm::BAR_OFF) + warp * NS * 8;
  float* psm = reinterpret_cast<float*>(smem + Gm::PSM_OFF) + warp * (32 + GP);
  const int32_t* bt = PAGED ? c.block_table + static_cast<int64_t>(b) * c.bt_stride : nullptr;

  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const uint64_t policy = l2_evict_first_policy();
  auto issue = [&](int it) {
    const int stg = it % NS;
    const int t0 = k0 + (warp + it * kWarps) * KT;
    const int cnt = min(KT, k1 - t0);
    const uint32_t bar = bar0 + 8 * stg;
    const uint32_t kd = smem_addr(wsm + stg * Gm::STAGE);
    const uint32_t vd = kd + Gm::TILE;
    mbar_arrive_expect_tx(bar, 2u * cnt * Gm::ROW);
    if constexpr (PAGED) {
      int t = t0, done = 0;
      while (t < t0 + cnt) {
        const int pi = t / c.P;
        const int off = t - pi * c.P;
        int pg = bt[pi];
        if (pg < 0 || pg >= c.n_rows) {
          raise_error(a.err, ERR_INDEX);
          pg = 0;
        }
        const int run = min(c.P - off, t0 + cnt - t);
        const int64_t src = ((static_cast<int64_t>(pg) * Hkv + j) * c.P + off) * D;
        bulk_copy_g2s(kd + done * Gm::ROW, sk.kb + src, run * Gm::ROW, bar, policy);
        bulk_copy_g2s(vd + done * Gm::ROW, sk.vb + src, run * Gm::ROW, bar, policy);
        t += run;
        done += run;
      }
    } else {
      int phys = sk.start + t0;
      if (phys >= c.R) phys -= c.R;
      const int run1 = min(cnt, c.R - phys);
      bulk_copy_g2s(kd, sk.kb + static_cast<int64_t>(phys) * D, run1 * Gm::ROW, bar, policy);
      bulk_copy_g2s(vd, sk.vb + static_cast<int64_t>(phys) * D, run1 * Gm::ROW, bar, policy);
      if (run1 < cnt) {
        bulk_copy_g2s(kd + run1 * Gm::ROW, sk.kb, (cnt - run1) * Gm::ROW, bar, policy);
        bulk_copy_g2s(vd + run1 * Gm::ROW, sk.vb, (cnt - run1) * Gm::ROW, bar, policy);
      }
    }
  };
  if (lane == 0) {
    const int pre = my_tiles < NS ? my_tiles : NS;
    for (int it = 0; it < pre; ++it) issue(it);
  }

  pdl_wait();  // the rotated, pre-scaled q of this call
  pdl_trigger();

  // This lane's 8 dims of each query head of the group (padding heads are 0).
  const int dl = (lane % LPK) * 8;
  float q[GP][8];
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    if (g < G) {
      const float* src = a.qhat + (static_cast<int64_t>(b) * Hkv * G + j * G + g) * D + dl;
      const float4 x0 = *reinterpret_cast<const float4*>(src);
      const float4 x1 = *reinterpret_cast<const float4*>(src + 4);
      q[g][0] = x0.x; q[g][1] = x0.y; q[g][2] = x0.z; q[g][3] = x0.w;
      q[g][4] = x1.x; q[g][5] = x1.y; q[g][6] = x1.z; q[g][7] = x1.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) q[g][e] = 0.f;
    }
  }

  float o[GP][8];
#pragma unroll
  for (int g = 0; g < GP; ++g)
#pragma unroll
    for (int e = 0; e < 8; ++e) o[g][e] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;
  const int half = lane / LPK;                        // key of a warp-wide load held by this lane
  const int key_s = ((lane % LPK) / GP) * KPS + half; // tile key of this lane's score

  for (int it = 0; it < my_tiles; ++it) {
    const int stg = it % NS;
    if (!mbar_wait_bounded(bar0 + 8 * stg, (it / NS) & 1)) {
      if (lane == 0) raise_error(a.err, ERR_TIMEOUT);
      break;
    }
    const int t0 = k0 + (warp + it * kWarps) * KT;
    const int nvalid = min(KT, k1 - t0);
    const uint4* Ks = reinterpret_cast<const uint4*>(wsm + stg * Gm::STAGE);
    const uint4* Vs = Ks + Gm::TILE / 16;

    // scores: J loads of 8 dims, GP heads each, then the transposing reduction
    float sp[J * GP];
#pragma unroll
    for (int jj = 0; jj < J; ++jj) {
      float kf[8];
      unpack8(Ks[jj * 32 + lane], kf);
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        float acc = q[g][0] * kf[0];
#pragma unroll
        for (int e = 1; e < 8; ++e) acc = fmaf(q[g][e], kf[e], acc);
        sp[jj * GP + g] = acc;
      }
    }
    float s = transpose_reduce<LPK>(sp, lane);
    if (key_s >= nvalid) s = -INFINITY;

    // online softmax (base 2): every lane holds one (key, head) score
    float tmax = s;
#pragma unroll
    for (int w = GP; w < 32; w <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, w));
    const float m_new = fmaxf(m_run, tmax);
    const float corr = exp2_fast(m_run - m_new);
    const float p = exp2_fast(s - m_new);
    l_run = fmaf(l_run, corr, p);
    m_run = m_new;
    psm[lane] = p;
    if (lane < GP) psm[32 + lane] = corr;
    __syncwarp();

#pragma unroll
    for (int g = 0; g < GP; ++g) {
      const float cr = psm[32 + g];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[g][e] *= cr;
    }
    if (nvalid == KT) {
#pragma unroll
      for (int jj = 0; jj < J; ++jj) {
        float vf[8];
        unpack8(Vs[jj * 32 + lane], vf);
        const float* pp = psm + half * LPK + jj * GP;
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float pg = pp[g];
#pragma unroll
          for (int e = 0; e < 8; ++e) o[g][e] = fmaf(pg, vf[e], o[g][e]);
        }
      }
    } else {
#pragma unroll
      for (int jj = 0; jj < J; ++jj) {
        if (jj * KPS + half < nvalid) {
          float vf[8];
          unpack8(Vs[jj * 32 + lane], vf);
          const float* pp = psm + half * LPK + jj * GP;
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            const float pg = pp[g];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[g][e] = fmaf(pg, vf[e], o[g][e]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0 && it + NS < my_tiles) {
      fence_proxy_async_smem();
      issue(it + NS);
    }
  }

  // warp totals: l over the lanes holding the same head; o over the keys of a
  // warp-wide load held by different lane groups
#pragma unroll
  for (int w = GP; w < 32; w <<= 1) l_run += __shfl_xor_sync(kFull, l_run, w);
#pragma unroll
  for (int w = LPK; w < 32; w <<= 1)
#pragma unroll
    for (int g = 0; g < GP; ++g)
#pragma unroll
      for (int e = 0; e < 8; ++e) o[g][e] += __shfl_xor_sync(kFull, o[g][e], w);

  // merge the warps in shared memory (the stage buffers are idle now)
  __syncthreads();
  float* mo = reinterpret_cast<float*>(smem);        // [kWarps][GP][D]
  float* mm = mo + kWarps * GP * D;                  // [kWarps][GP]
  float* ml = mm + kWarps * GP;                      // [kWarps][GP]
  if (lane < LPK) {
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      float* dst = mo + (warp * GP + g) * D + dl;
      *reinterpret_cast<float4*>(dst) = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(o[g][4], o[g][5], o[g][6], o[g][7]);
    }
  }
  if (lane < GP) {
    mm[warp * GP + lane] = m_run;
    ml[warp * GP + lane] = l_run;
  }
  __syncthreads();
  float* dst = a.part + ((static_cast<int64_t>(b) * Hkv + j) * a.splits + split) * (GP * (D + 2));
  for (int e = threadIdx.x; e < GP * D; e += kWarps * 32) {
    const int g = e / D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mm[w * GP + g]);
    float acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) acc = fmaf(exp2_fast(mm[w * GP + g] - M), mo[(w * GP + g) * D + (e - g * D)], acc);
    }
    dst[e] = acc;
  }
  if (threadIdx.x < GP) {
    const int g = threadIdx.x;
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mm[w * GP + g]);
    float L = 0.f;
    if (M != -INFINITY)
      for (int w = 0; w < kWarps; ++w) L = fmaf(exp2_fast(mm[w * GP + g] - M), ml[w * GP + g], L);
    dst[GP * D + g] = M;
    dst[GP * D + GP + g] = L;
  }
}

// ---------------------------------------------------------------- combine

// Threads per head in the combine: TPH lanes, each 4 dims of a DSPLIT-th of D.
// One CTA per (dim chunk, KV head, stream); the G heads of the group each use
// TPH consecutive lanes of one warp.
template <int TPH>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int w = TPH / 2; w >= 1; w >>= 1) x += __shfl_xor_sync(kFull, x, w);
  return x;
}
template <int TPH>
__device__ __forceinline__ float group_max(float x) {
#pragma unroll
  for (int w = TPH / 2; w >= 1; w >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, w));
  return x;
}

template <int D, int TPH, bool PAGED>
__global__ void __launch_bounds__(256) decode_combine_kernel(const CombineArgs a, int G, int GP) {
  extern __shared__ float wsm[];  // [heads in block][splits]: weights of the splits
  const int chunk_d = TPH * 4;
  const int dc = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  // the block is a whole number of warps; lanes past the G heads repeat the
  // last head's arithmetic (for the shuffles) and store nothing
  const int gb = threadIdx.x / TPH, t = threadIdx.x % TPH;
  const bool active = gb < G;
  const int g = active ? gb : G - 1;
  const int d4 = dc * chunk_d + t * 4;
  const int Hkv = a.Hkv, Hq = Hkv * G, h = j * G + g;
  const CacheView& c = a.c;

  // ---- caller inputs (not produced by the split kernel): before the wait
  int n = 0, wb_slot = -1;
  int64_t wb_off = -1;  // element offset of the new entry's row for KV head j
  if constexpr (PAGED) {
    n = c.seq_len[b];
    const int cap = min(a.max_len, c.bt_stride * c.P);
    n = n < 0 ? 0 : (n > cap ? cap : n);
    if (a.write_back) {
      const int pi = n / c.P;
      const int pg = pi < c.bt_stride ? c.block_table[static_cast<int64_t>(b) * c.bt_stride + pi] : -1;
      if (pg >= 0 && pg < c.n_rows)
        wb_off = ((static_cast<int64_t>(pg) * Hkv + j) * c.P + n % c.P) * D;
      else if (dc == 0 && threadIdx.x == 0)
        raise_error(a.err, ERR_INDEX);
    }
  } else {
    const int row = c.stream_rows ? c.stream_rows[b] : b;
    const int head = c.ring_head[b], cnt = c.ring_count[b];
    if (!(row < 0 || row >= c.n_rows || head < 0 || head >= c.R || cnt < 0 || cnt > c.R)) {
      n = cnt;
      wb_slot = head;
      wb_off = ((static_cast<int64_t>(row) * Hkv + j) * c.R + wb_slot) * D;
    }
  }
  const int S = n > 0 ? (n + a.chunk - 1) / a.chunk : 0;
  const uint2 vw = *reinterpret_cast<const uint2*>(a.v_new + (static_cast<int64_t>(b) * Hkv + j) * D + d4);
  float sig = 1.f;
  if (a.gate) sig = 1.f / (1.f + expf(-bf16_to_f32(a.gate[static_cast<int64_t>(b) * Hq + h])));

  pdl_wait();  // partials of the split kernel
  pdl_trigger();

  // ---- new token's score (base 2): q_hat (pre-scaled) . k_entry over all D
  const float* qh = a.qhat + (static_cast<int64_t>(b) * Hq + h) * D;
  const uint16_t* kh = a.khat + (static_cast<int64_t>(b) * Hkv + j) * D;
  float dot = 0.f;
  for (int d = t * 4; d < D; d += TPH * 4) {
    const float4 qv = *reinterpret_cast<const float4*>(qh + d);
    const uint2 kw = *reinterpret_cast<const uint2*>(kh + d);
    dot = fmaf(qv.x, bf16_lo(kw.x), dot);
    dot = fmaf(qv.y, bf16_hi(kw.x), dot);
    dot = fmaf(qv.z, bf16_lo(kw.y), dot);
    dot = fmaf(qv.w, bf16_hi(kw.y), dot);
  }
  const float s_new = group_sum<TPH>(dot);

  // ---- merge: M over the splits and the new token, then weights and L
  const int stride = GP * (D + 2);
  const float* P0 = a.part + (static_cast<int64_t>(b) * Hkv + j) * a.splits * stride;
  float M = s_new;
  for (int s = t; s < S; s += TPH) M = fmaxf(M, P0[s * stride + GP * D + g]);
  M = group_max<TPH>(M);
  float L = 0.f;
  for (int s = t; s < S; s += TPH) {
    const float w = exp2_fast(P0[s * stride + GP * D + g] - M);
    wsm[gb * a.splits + s] = w;
    L = fmaf(w, P0[s * stride + GP * D + GP + g], L);
  }
  L = group_sum<TPH>(L);
  __syncwarp();
  // the weighted sum of the partial outputs: loads issued ahead of the FMAs
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* po = P0 + g * D + d4;
  int s = 0;
  for (; s + 4 <= S; s += 4) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = *reinterpret_cast<const float4*>(po + (s + u) * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = wsm[gb * a.splits + s + u];
      acc.x = fmaf(w, v[u].x, acc.x);
      acc.y = fmaf(w, v[u].y, acc.y);
      acc.z = fmaf(w, v[u].z, acc.z);
      acc.w = fmaf(w, v[u].w, acc.w);
    }
  }
  for (; s < S; ++s) {
    const float4 v = *reinterpret_cast<const float4*>(po + s * stride);
    const float w = wsm[gb * a.splits + s];
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  // the new token joins as a length-1 score vector
  const float wn = exp2_fast(s_new - M);
  L += wn;
  acc.x = fmaf(wn, bf16_lo(vw.x), acc.x);
  acc.y = fmaf(wn, bf16_hi(vw.x), acc.y);
  acc.z = fmaf(wn, bf16_lo(vw.y), acc.z);
  acc.w = fmaf(wn, bf16_hi(vw.y), acc.w);
  if (!active) return;
  const float scale = sig / L;
  *reinterpret_cast<float4*>(a.out + (static_cast<int64_t>(b) * Hq + h) * D + d4) =
      make_float4(acc.x * scale, acc.y * scale, acc.z * scale, acc.w * scale);

  // ---- write-back of the new entry, after every read of the cache (the split
  // kernel has completed): the rotated bf16 key and the value
  if (a.write_back && g == 0 && wb_off >= 0) {
    *reinterpret_cast<uint2*>(c.k + wb_off + d4) = *reinterpret_cast<const uint2*>(kh + d4);
    *reinterpret_cast<uint2*>(c.v + wb_off + d4) = vw;
  }
}

template <int D, int GP, bool PAGED>
cudaError_t split_launch(const SplitArgs& a, int G, cudaStream_t s) {
  using Gm = Geo<D, GP>;
  auto k = decode_split_kernel<D, GP, PAGED>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(a.splits, a.Hkv, a.B);
  return launch_pdl(k, grid, dim3(kWarps * 32), Gm::SMEM, s, a, G);
}

template <int D, int GP>
cudaError_t split_dispatch_paged(const SplitArgs& a, int G, cudaStream_t s) {
  return a.c.paged ? split_launch<D, GP, true>(a, G, s) : split_launch<D, GP, false>(a, G, s);
}

int padded_group(int G) { return G <= 2 ? 2 : (G <= 4 ? 4 : (G <= 8 ? 8 : 0)); }

}  // namespace

cudaError_t launch_decode_split(const SplitArgs& a, int D, int G, cudaStream_t s) {
  const int GP = padded_group(G);
  if (D == 256) {
    if (GP == 2) return split_dispatch_paged<256, 2>(a, G, s);
    if (GP == 4) return split_dispatch_paged<256, 4>(a, G, s);
    if (GP == 8) return split_dispatch_paged<256, 8>(a, G, s);
  } else if (D == 128) {
    if (GP == 2) return split_dispatch_paged<128, 2>(a, G, s);
    if (GP == 4) return split_dispatch_paged<128, 4>(a, G, s);
    if (GP == 8) return split_dispatch_paged<128, 8>(a, G, s);
  }
  return cudaErrorNotSupported;
}

int decode_split_tile_keys(int D, int G) {
  const int GP = padded_group(G);
  if (GP == 0 || (D != 128 && D != 256)) return 0;
  return (D / 8 / GP) * (32 / (D / 8));
}

int decode_split_ctas_per_sm(int D, int G) {
  const int GP = padded_group(G);
  int smem = 0;
  if (D == 256) smem = GP == 2 ? Geo<256, 2>::SMEM : GP == 4 ? Geo<256, 4>::SMEM : GP == 8 ? Geo<256, 8>::SMEM : 0;
  if (D == 128) smem = GP == 2 ? Geo<128, 2>::SMEM : GP == 4 ? Geo<128, 4>::SMEM : GP == 8 ? Geo<128, 8>::SMEM : 0;
  if (smem == 0) return 0;
  // 228 KB of shared memory per SM, 1 KB of it reserved per resident CTA
  int per_sm = (233472) / (smem + 1024);
  return per_sm > 2 ? 2 : per_sm;
}

cudaError_t launch_decode_combine(const CombineArgs& a, int D, int G, cudaStream_t s) {
  const int GP = padded_group(G);
  if (GP == 0) return cudaErrorNotSupported;
  // dims per CTA: enough CTAs to spread the partial reads, at most 32 lanes per head
  const int units = a.B * a.Hkv;
  int dsplit = (152 + units - 1) / units;
  const int dmin = D / 128;  // TPH <= 32
  const int dmax = D / 32;   // TPH >= 8
  dsplit = dsplit < dmin ? dmin : (dsplit > dmax ? dmax : dsplit);
  // round up to a power of two
  int p2 = 1;
  while (p2 < dsplit) p2 <<= 1;
  dsplit = p2 > dmax ? dmax : p2;
  const int tph = D / 4 / dsplit;
  dim3 grid(dsplit, a.Hkv, a.B);
  const int threads = (G * tph + 31) / 32 * 32;
  dim3 block(threads);
  const size_t smem = static_cast<size_t>(threads / tph) * a.splits * sizeof(float);
  const bool paged = a.c.paged != 0;
#define DATTN_COMBINE(DD, TT)                                                                     \
  if (D == DD && tph == TT)                                                                       \
    return paged ? launch_pdl(decode_combine_kernel<DD, TT, true>, grid, block, smem, s, a, G, GP) \
                 : launch_pdl(decode_combine_kernel<DD, TT, false>, grid, block, smem, s, a, G, GP);
  DATTN_COMBINE(256, 32)
  DATTN_COMBINE(256, 16)
  DATTN_COMBINE(256, 8)
  DATTN_COMBINE(128, 32)
  DATTN_COMBINE(128, 16)
  DATTN_COMBINE(128, 8)
#undef DATTN_COMBINE
  return cudaErrorNotSupported;
}

}  // namespace dattn
