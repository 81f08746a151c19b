// Decode attention: the split-K pass over the cached keys and the LSE combine
// that joins the new token in score space.
//
// Method ("vllm-omni commits", score-space join commit): the cached keys (n of
// them) and the new key are scored separately and their score vectors meet in
// one softmax; nothing cache-sized is copied, and the new K/V entry is written
// into its slot afterwards. A ring's slots need no reordering (softmax is
// order-free, cached keys carry their own rotary phase); unwritten slots are
// masked by never being read. Grouped-query attention shares each KV head's
// loads among its G query heads ("vllm-omni commits", talker export commit).
// Splitting the keys over many CTAs and merging their partial softmax states
// follows "TensorFold PR #608" (the split "shared" kernel plus a merge, the
// lessons that the grid must fill the GPU and that a merge must not be a chain
// of dependent loads).
//
// GB300 design.
//  * Work split (stream-K). A "unit" is one (stream, KV head); its cached keys
//    form ceil(n / SK) stage tiles. All units' tiles are laid end to end and the
//    grid - exactly the CTAs that fit on the GPU at once - cuts that sequence
//    into equal contiguous ranges, so every CTA moves the same number of bytes
//    whatever the mix of lengths. Each piece of a unit inside one CTA (a
//    "segment") leaves one partial softmax state (m, l, o); the combine merges
//    a unit's segments.
//  * Loads. Each warp owns a private ring of NS stage buffers. One lane issues
//    bulk TMA copies (cp.async.bulk global -> shared, completion counted in
//    transaction bytes on the stage's mbarrier) for the K and V rows of the
//    warp's tile NS ahead; the ring keeps streaming across segment boundaries.
//    Pages and ring wrap-around turn into one copy per contiguous run of rows.
//  * Math. At G flops per byte the KV stream is HBM-bound, so scores and the
//    value sum run on the FP32 pipes. A lane holds 8 dims (one 16-byte shared
//    load) of a key; the per-head dot products of J keys are reduced across the
//    lanes of a key by a transposing butterfly that leaves exactly one
//    (key, head) score per lane, so the online softmax costs one exp2 per lane
//    per sub-tile. Probabilities reach all lanes through shared memory.
#include "common.cuh"

namespace dattn {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxUnits = 1024;   // (stream, KV head) units per call

template <int D, int GP>
struct Geo {
  static constexpr int LPK = D / 8;          // lanes per key row (16 bytes each)
  static constexpr int KPS = 32 / LPK;       // keys per warp-wide load
  static constexpr int J = LPK / GP;         // loads per sub-tile (J * GP scores per lane)
  static constexpr int KT = J * KPS;         // keys per sub-tile
  static constexpr int ROW = D * 2;          // bytes per key row
  static constexpr int SK_MIN = 8192 / (2 * ROW);
  static constexpr int SUB = KT >= SK_MIN ? 1 : SK_MIN / KT;
  static constexpr int SK = KT * SUB;        // keys per stage tile (>= 8 KB of K + V)
  static constexpr int TILE = SK * ROW;      // bytes of the K (or V) half of a stage
  static constexpr int STAGE = 2 * TILE;
  static constexpr int NS = STAGE >= 16384 ? 2 : 3;
  static constexpr int BAR_OFF = kWarps * NS * STAGE;
  static constexpr int ML_OFF = BAR_OFF + kWarps * NS * 8;     // float [kWarps][2*GP]
  static constexpr int SLOT_OFF = ML_OFF + kWarps * 2 * GP * 4; // int [kWarps]
  static constexpr int PSM_OFF = SLOT_OFF + kWarps * 4;         // float [kWarps][32+GP]
  static constexpr int TAB_OFF = (PSM_OFF + kWarps * (32 + GP) * 4 + 15) / 16 * 16;
  static constexpr int SMEM_MAX = TAB_OFF + (2 * kMaxUnits + 1) * 4;
  static_assert(D == 128 || D == 256, "head_dim");
  static_assert(LPK % GP == 0, "GP must divide the lanes per key");
  static_assert(GP * D * 4 <= STAGE, "a stage buffer holds one warp's partial output");
};

__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
  f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x);
  f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
  f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z);
  f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
}

__device__ __forceinline__ void unpack8x2(const uint4& w, float2 (&f)[4]) {
  f[0] = make_float2(bf16_lo(w.x), bf16_hi(w.x));
  f[1] = make_float2(bf16_lo(w.y), bf16_hi(w.y));
  f[2] = make_float2(bf16_lo(w.z), bf16_hi(w.z));
  f[3] = make_float2(bf16_lo(w.w), bf16_hi(w.w));
}

// Sum W partial values across W lanes (W a power of two, groups aligned) so
// that lane l ends with the full sum of value (l % W). At each level the lane
// whose bit `w` is set keeps the upper half of its values and sends the lower
// half to its partner, which does the opposite.
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

// Cached keys of call row b (the same for all its KV heads). Bad metadata is
// reported (once per row) and yields no keys.
template <bool PAGED>
__device__ __forceinline__ int unit_length(const CacheView& c, int b, int max_len, bool report,
                                           int* err) {
  if constexpr (PAGED) {
    int n = c.seq_len[b];
    const int cap = min(max_len, c.bt_stride * c.P);
    if (n < 0 || n > cap) {
      if (report) raise_error(err, ERR_LENGTH);
      n = n < 0 ? 0 : cap;
    }
    return n;
  } else {
    const int row = c.stream_rows ? c.stream_rows[b] : b;
    const int head = c.ring_head[b], cnt = c.ring_count[b];
    if (row < 0 || row >= c.n_rows || head < 0 || head >= c.R || cnt < 0 || cnt > c.R) {
      if (report) raise_error(err, ERR_INDEX);
      return 0;
    }
    return cnt;
  }
}

template <int D, int GP, bool PAGED>
__global__ void __launch_bounds__(kThreads, 2) decode_split_kernel(const SplitArgs a, int G) {
  using Gm = Geo<D, GP>;
  constexpr int LPK = Gm::LPK, KPS = Gm::KPS, J = Gm::J, KT = Gm::KT, SK = Gm::SK;
  constexpr int SUB = Gm::SUB, NS = Gm::NS;
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const CacheView& c = a.c;
  const int Hkv = a.Hkv, U = a.B * Hkv;
  const int NC = gridDim.x, cta = blockIdx.x;
  int* P = reinterpret_cast<int*>(smem + Gm::TAB_OFF);  // [U + 1] tile prefix over units
  int* N = P + U + 1;                                    // [U] cached keys per unit

  // ---- unit table from caller metadata (not written by the preceding kernel)
  for (int u = threadIdx.x; u < U; u += kThreads) {
    const int b = u / Hkv;
    const int n = unit_length<PAGED>(c, b, a.max_len, cta == 0 && u - b * Hkv == 0, a.err);
    N[u] = n;
    P[u + 1] = (n + SK - 1) / SK;
  }
  if (threadIdx.x == 0) P[0] = 0;
  __syncthreads();
  block_scan_inclusive<kThreads>(P + 1, U);
  const int T = P[U];
  const int g0 = static_cast<int>(static_cast<int64_t>(cta) * T / NC);
  const int g1 = static_cast<int>(static_cast<int64_t>(cta + 1) * T / NC);
  if (cta == 0)  // the combine locates each unit's segments from this table
    for (int u = threadIdx.x; u <= U; u += kThreads) a.tiles[u] = P[u];

  // ---- this warp's tiles: g = g0 + warp + kWarps * it
  const int span = g1 - g0;
  const int my_n = span > warp ? (span - warp + kWarps - 1) / kWarps : 0;
  uint8_t* wsm = smem + warp * NS * Gm::STAGE;
  const uint32_t bar0 = smem_addr(smem + Gm::BAR_OFF) + warp * NS * 8;
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const uint64_t policy = l2_evict_first_policy();
  int u_iss = my_n > 0 ? unit_of(P, U, g0 + warp) : 0;
  // Request tile `it` of this warp into stage it % NS (one lane).
  auto issue = [&](int it) {
    const int g = g0 + warp + kWarps * it;
    while (P[u_iss + 1] <= g) ++u_iss;
    const int u = u_iss;
    const int b = u / Hkv, j = u - b * Hkv;
    const int k0 = (g - P[u]) * SK;
    const int cnt = min(SK, N[u] - k0);
    const uint32_t bar = bar0 + 8 * (it % NS);
    const uint32_t kd = smem_addr(wsm + (it % NS) * Gm::STAGE);
    const uint32_t vd = kd + Gm::TILE;
    mbar_arrive_expect_tx(bar, 2u * cnt * Gm::ROW);
    if constexpr (PAGED) {
      const int32_t* bt = c.block_table + static_cast<int64_t>(b) * c.bt_stride;
      int t = k0, done = 0;
      while (t < k0 + cnt) {
        const int pi = t / c.P;
        const int off = t - pi * c.P;
        int pg = bt[pi];
        if (pg < 0 || pg >= c.n_rows) {
          raise_error(a.err, ERR_INDEX);
          pg = 0;
        }
        const int run = min(c.P - off, k0 + cnt - t);
        const int64_t src = ((static_cast<int64_t>(pg) * Hkv + j) * c.P + off) * D;
        bulk_copy_g2s(kd + done * Gm::ROW, c.k + src, run * Gm::ROW, bar, policy);
        bulk_copy_g2s(vd + done * Gm::ROW, c.v + src, run * Gm::ROW, bar, policy);
        t += run;
        done += run;
      }
    } else {
      const int row = c.stream_rows ? c.stream_rows[b] : b;
      const int n = N[u];
      const int head = c.ring_head[b];
      const int start = head - n < 0 ? head - n + c.R : head - n;
      const int64_t base = (static_cast<int64_t>(row) * Hkv + j) * c.R * D;
      int phys = start + k0;
      if (phys >= c.R) phys -= c.R;
      const int run1 = min(cnt, c.R - phys);
      bulk_copy_g2s(kd, c.k + base + static_cast<int64_t>(phys) * D, run1 * Gm::ROW, bar, policy);
      bulk_copy_g2s(vd, c.v + base + static_cast<int64_t>(phys) * D, run1 * Gm::ROW, bar, policy);
      if (run1 < cnt) {
        bulk_copy_g2s(kd + run1 * Gm::ROW, c.k + base, (cnt - run1) * Gm::ROW, bar, policy);
        bulk_copy_g2s(vd + run1 * Gm::ROW, c.v + base, (cnt - run1) * Gm::ROW, bar, policy);
      }
    }
  };
  if (lane == 0) {
    const int pre = my_n < NS ? my_n : NS;
    for (int it = 0; it < pre; ++it) issue(it);
  }

  pdl_wait();  // the rotated, pre-scaled q of this call
  pdl_trigger();

  float* ML = reinterpret_cast<float*>(smem + Gm::ML_OFF);
  int* SLOT = reinterpret_cast<int*>(smem + Gm::SLOT_OFF);
  float* psm = reinterpret_cast<float*>(smem + Gm::PSM_OFF) + warp * (32 + GP);
  const int dl = (lane % LPK) * 8;
  const int half = lane / LPK;                         // key of a warp-wide load held by this lane
  const int key_s = ((lane % LPK) / GP) * KPS + half;  // sub-tile key of this lane's score

  bool failed = false;
  int it = 0;
  int deferred = -1;
  bool first_seg = true;
  for (int u = span > 0 ? unit_of(P, U, g0) : U; u < U && P[u] < g1; ++u) {
    if (P[u + 1] == P[u]) continue;  // a unit with no cached keys
    const int ge = min(g1, P[u + 1]);
    const int b = u / Hkv, j = u - b * Hkv;

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
    int last_stage = -1;

    for (;;) {
      const int g = g0 + warp + kWarps * it;
      if (it >= my_n || g >= ge) break;
      const int stg = it % NS;
      if (!failed) {
        // the whole warp agrees on the outcome, so the shuffles below stay converged
        const bool ok = __all_sync(kFull, mbar_wait_bounded(bar0 + 8 * stg, (it / NS) & 1));
        if (!ok) {
          failed = true;
          if (lane == 0) raise_error(a.err, ERR_TIMEOUT);
        }
      }
      if (!failed) {
        const int nstage = min(SK, N[u] - (g - P[u]) * SK);
#pragma unroll 1
        for (int sb = 0; sb < SUB; ++sb) {
          const int nvalid = nstage - sb * KT;
          if (nvalid <= 0) break;
          const uint4* Ks = reinterpret_cast<const uint4*>(wsm + stg * Gm::STAGE) + sb * (KT * D / 8);
          const uint4* Vs = Ks + Gm::TILE / 16;

          // scores: J loads of 8 dims for GP heads, then the transposing reduction
          float sp[J * GP];
#pragma unroll
          for (int jj = 0; jj < J; ++jj) {
            float kf[8];
            unpack8(Ks[jj * 32 + lane], kf);
#pragma unroll
            for (int h = 0; h < GP; ++h) {
              float acc = q[h][0] * kf[0];
#pragma unroll
              for (int e = 1; e < 8; ++e) acc = fmaf(q[h][e], kf[e], acc);
              sp[jj * GP + h] = acc;
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
          for (int h = 0; h < GP; ++h) {
            const float cr = psm[32 + h];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[h][e] *= cr;
          }
          if (nvalid >= KT) {
#pragma unroll
            for (int jj = 0; jj < J; ++jj) {
              float vf[8];
              unpack8(Vs[jj * 32 + lane], vf);
              const float* pp = psm + half * LPK + jj * GP;
#pragma unroll
              for (int h = 0; h < GP; ++h) {
                const float ph = pp[h];
#pragma unroll
                for (int e = 0; e < 8; ++e) o[h][e] = fmaf(ph, vf[e], o[h][e]);
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
                for (int h = 0; h < GP; ++h) {
                  const float ph = pp[h];
#pragma unroll
                  for (int e = 0; e < 8; ++e) o[h][e] = fmaf(ph, vf[e], o[h][e]);
                }
              }
            }
          }
          __syncwarp();
        }
      }
      last_stage = stg;
      // Refill this stage with the warp's tile NS ahead. The warp's last tile
      // of a segment keeps its stage as the merge buffer until the merge is done.
      if (it + NS < my_n) {
        if (g + kWarps >= ge) {
          deferred = it + NS;
        } else if (lane == 0 && !failed) {
          fence_proxy_async_smem();
          issue(it + NS);
        }
      }
      ++it;
    }

    // ---- merge the warps' states for this segment
#pragma unroll
    for (int w = GP; w < 32; w <<= 1) l_run += __shfl_xor_sync(kFull, l_run, w);
#pragma unroll
    for (int w = LPK; w < 32; w <<= 1)
#pragma unroll
      for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) o[h][e] += __shfl_xor_sync(kFull, o[h][e], w);
    if (last_stage >= 0 && lane < LPK) {
      float* os = reinterpret_cast<float*>(wsm + last_stage * Gm::STAGE);
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        *reinterpret_cast<float4*>(os + h * D + dl) = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
        *reinterpret_cast<float4*>(os + h * D + dl + 4) = make_float4(o[h][4], o[h][5], o[h][6], o[h][7]);
      }
    }
    if (lane < GP) {
      ML[warp * 2 * GP + lane] = last_stage >= 0 ? m_run : -INFINITY;
      ML[warp * 2 * GP + GP + lane] = last_stage >= 0 ? l_run : 0.f;
    }
    if (lane == 0) SLOT[warp] = last_stage;
    __syncthreads();
    const int slot = first_seg ? cta : NC + u;
    float* dst = a.part + static_cast<int64_t>(slot) * (GP * (D + 2));
    for (int e = threadIdx.x; e < GP * D; e += kThreads) {
      const int h = e / D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ML[w * 2 * GP + h]);
      float acc = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const int st = SLOT[w];
          if (st >= 0) {
            const float* os = reinterpret_cast<const float*>(smem + (w * NS + st) * Gm::STAGE);
            acc = fmaf(exp2_fast(ML[w * 2 * GP + h] - M), os[e], acc);
          }
        }
      }
      dst[e] = acc;
    }
    if (threadIdx.x < GP) {
      const int h = threadIdx.x;
      float M = -INFINITY;
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ML[w * 2 * GP + h]);
      float L = 0.f;
      if (M != -INFINITY)
        for (int w = 0; w < kWarps; ++w) L = fmaf(exp2_fast(ML[w * 2 * GP + h] - M), ML[w * 2 * GP + GP + h], L);
      dst[GP * D + h] = M;
      dst[GP * D + GP + h] = L;
    }
    __syncthreads();
    if (deferred >= 0) {
      if (lane == 0 && !failed) {
        fence_proxy_async_smem();
        issue(deferred);
      }
      deferred = -1;
    }
    first_seg = false;
  }
}

// ---------------------------------------------------------------- combine

// One CTA per (dim chunk, KV head, stream); the G heads of the group each use
// TPH consecutive lanes of one warp, 4 dims per lane.
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
  extern __shared__ float wsm[];  // [heads in block][max segments]: merge weights
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
  int64_t wb_off = -1;  // element offset of the new entry's row for KV head j
  if constexpr (PAGED) {
    int n = c.seq_len[b];
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
    if (!(row < 0 || row >= c.n_rows || head < 0 || head >= c.R || cnt < 0 || cnt > c.R))
      wb_off = ((static_cast<int64_t>(row) * Hkv + j) * c.R + head) * D;
  }
  const uint2 vw = *reinterpret_cast<const uint2*>(a.v_new + (static_cast<int64_t>(b) * Hkv + j) * D + d4);
  float sig = 1.f;
  if (a.gate) sig = 1.f / (1.f + expf(-bf16_to_f32(a.gate[static_cast<int64_t>(b) * Hq + h])));

  pdl_wait();  // partials and the tile table of the split kernel
  pdl_trigger();

  // ---- this unit's segments: CTAs c_lo..c_hi of the split grid
  const int U = a.B * Hkv, u = b * Hkv + j, NC = a.split_ctas;
  const int T = a.tiles[U];
  const int p0 = a.tiles[u], p1 = a.tiles[u + 1];
  int S = 0, c_lo = 0, first_slot = 0;
  if (p1 > p0) {
    // CTA of global tile x: floor(((x + 1) * NC - 1) / T)
    c_lo = static_cast<int>((static_cast<int64_t>(p0 + 1) * NC - 1) / T);
    const int c_hi = static_cast<int>((static_cast<int64_t>(p1) * NC - 1) / T);
    S = c_hi - c_lo + 1;
    const int begin_lo = static_cast<int>(static_cast<int64_t>(c_lo) * T / NC);
    first_slot = begin_lo == p0 ? c_lo : NC + u;
  }

  // ---- loads first: the segments' (m, l) and their first output slices,
  // q_hat and the new key entry - none depends on another
  const int stride = GP * (D + 2);
  auto seg = [&](int k) -> const float* {
    return a.part + static_cast<int64_t>(k == 0 ? first_slot : c_lo + k) * stride;
  };
  // Segment k > 0 is the first segment of split CTA c_lo + k - unless that CTA
  // got no tiles at all (possible when the call's keys are far below its
  // planned bound), in which case it wrote nothing and is skipped.
  auto seg_ok = [&](int k) -> bool {
    if (k == 0) return true;
    const int64_t cc = c_lo + k;
    return cc * T / NC < (cc + 1) * T / NC;
  };
  constexpr int kPre = 4;
  float mk = -INFINITY, lk = 0.f;
  if (t < S && seg_ok(t)) {
    const float* pk = seg(t);
    mk = pk[GP * D + g];
    lk = pk[GP * D + GP + g];
  }
  float4 ov[kPre];
#pragma unroll
  for (int x = 0; x < kPre; ++x)
    ov[x] = x < S && seg_ok(x) ? *reinterpret_cast<const float4*>(seg(x) + g * D + d4)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int NQ = D / (4 * TPH);
  const float* qh = a.qhat + (static_cast<int64_t>(b) * Hq + h) * D;
  const uint16_t* kh = a.khat + (static_cast<int64_t>(b) * Hkv + j) * D;
  float4 qv[NQ];
  uint2 kv[NQ];
#pragma unroll
  for (int x = 0; x < NQ; ++x) {
    qv[x] = *reinterpret_cast<const float4*>(qh + (t + x * TPH) * 4);
    kv[x] = *reinterpret_cast<const uint2*>(kh + (t + x * TPH) * 4);
  }

  // ---- new token's score (base 2): q_hat (pre-scaled) . k_entry over all D
  float dot = 0.f;
#pragma unroll
  for (int x = 0; x < NQ; ++x) {
    dot = fmaf(qv[x].x, bf16_lo(kv[x].x), dot);
    dot = fmaf(qv[x].y, bf16_hi(kv[x].x), dot);
    dot = fmaf(qv[x].z, bf16_lo(kv[x].y), dot);
    dot = fmaf(qv[x].w, bf16_hi(kv[x].y), dot);
  }
  const float s_new = group_sum<TPH>(dot);

  // ---- merge: M over the segments and the new token, weights, L, outputs
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto fold = [&](float w, const float4& v) {
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  };
  float M, L;
  if (S <= TPH) {
    // one segment per lane: weights stay in registers and are broadcast
    M = group_max<TPH>(fmaxf(s_new, mk));
    const float w = t < S ? exp2_fast(mk - M) : 0.f;
    L = group_sum<TPH>(w * lk);
    const int base = threadIdx.x - t;  // first lane of this head's group
#pragma unroll
    for (int x = 0; x < kPre; ++x) {
      const float wx = __shfl_sync(kFull, w, (base + x) & 31);
      if (x < S) fold(wx, ov[x]);
    }
    for (int k = kPre; k < S; ++k) {
      const float wk = __shfl_sync(kFull, w, (base + k) & 31);
      if (seg_ok(k)) fold(wk, *reinterpret_cast<const float4*>(seg(k) + g * D + d4));
    }
  } else {
    M = mk;
    for (int k = t + TPH; k < S; k += TPH)
      if (seg_ok(k)) M = fmaxf(M, seg(k)[GP * D + g]);
    M = group_max<TPH>(fmaxf(M, s_new));
    L = 0.f;
    for (int k = t; k < S; k += TPH) {
      float w = 0.f;
      if (seg_ok(k)) {
        const float* pk = seg(k);
        w = exp2_fast(pk[GP * D + g] - M);
        L = fmaf(w, pk[GP * D + GP + g], L);
      }
      wsm[gb * a.split_ctas + k] = w;
    }
    L = group_sum<TPH>(L);
    __syncwarp();
#pragma unroll
    for (int x = 0; x < kPre; ++x) fold(wsm[gb * a.split_ctas + x], ov[x]);
    for (int k = kPre; k < S; ++k)
      if (seg_ok(k)) fold(wsm[gb * a.split_ctas + k], *reinterpret_cast<const float4*>(seg(k) + g * D + d4));
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

// ---------------------------------------------------------------- one-launch decode

template <int D, int GP>
struct FGeo {
  using Gm = Geo<D, GP>;
  static constexpr int QS_OFF = Gm::TAB_OFF;                    // float [GP][D]: rotated q of the unit
  static constexpr int SN_OFF = QS_OFF + GP * D * 4;            // float [GP]: new-token scores
  static constexpr int FLAG_OFF = SN_OFF + GP * 4;              // int: "this CTA combines"
  static constexpr int TAB_OFF = (FLAG_OFF + 4 + 15) / 16 * 16;  // int P[U+1], N[U]
  static constexpr int SMEM_MAX = TAB_OFF + (2 * kMaxUnits + 1) * 4;
};

// Rotate the G query heads of unit (b, j) into qs[GP][D] (fp32, pre-scaled;
// heads >= G are zero). All threads of the CTA take part, one pair at a time,
// each pair's cos and sin shared by the heads.
template <int D, int GP>
__device__ __forceinline__ void fused_rope_q(const FusedArgs& a, int b, int j, float* qs) {
  const int G = a.G, Hq = a.Hkv * G, half = a.r / 2;
  const int64_t pos = a.pos[b];
  const uint16_t* src = a.q + (static_cast<int64_t>(b) * Hq + j * G) * D;
  for (int p = threadIdx.x; p < D / 2; p += kThreads) {
    const int d0 = p < half ? p : a.r + 2 * (p - half);
    const int d1 = p < half ? p + half : d0 + 1;
    float c = 1.f, s = 0.f;
    if (p < half) rope_cos_sin(pos, a.rope_step[p], c, s);
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      float o0 = 0.f, o1 = 0.f;
      if (g < G) {
        const float x = bf16_to_f32(src[g * D + d0]), y = bf16_to_f32(src[g * D + d1]);
        if (p < half) {
          o0 = fmaf(x, c, -y * s) * a.q_scale;
          o1 = fmaf(y, c, x * s) * a.q_scale;
        } else {
          o0 = x * a.q_scale;
          o1 = y * a.q_scale;
        }
      }
      qs[g * D + d0] = o0;
      qs[g * D + d1] = o1;
    }
  }
}

// The bit-exact K entry of unit (b, j): bf16_RNE(x*c - y*s) evaluated in fp64
// (both products exact, one rounding) with the fp32 cos and sin of
// rope_cos_sin. Written to the workspace.
template <int D>
__device__ __forceinline__ void fused_k_entry(const FusedArgs& a, int b, int j, uint16_t* dst) {
  const int half = a.r / 2;
  const uint16_t* src = a.k_new + (static_cast<int64_t>(b) * a.Hkv + j) * D;
  const int64_t pos = a.pos[b];
  for (int p = threadIdx.x; p < D / 2; p += kThreads) {
    const int d0 = p < half ? p : a.r + 2 * (p - half);
    const int d1 = p < half ? p + half : d0 + 1;
    if (p < half) {
      float cf, sf;
      rope_cos_sin(pos, a.rope_step[p], cf, sf);
      const double c64 = cf, s64 = sf;
      const double x = bf16_to_f32(src[d0]), y = bf16_to_f32(src[d1]);
      dst[d0] = f64_to_bf16(__dsub_rn(__dmul_rn(x, c64), __dmul_rn(y, s64)));
      dst[d1] = f64_to_bf16(__dadd_rn(__dmul_rn(y, c64), __dmul_rn(x, s64)));
    } else {
      dst[d0] = src[d0];
      dst[d1] = src[d1];
    }
  }
}

// Number of split CTAs whose ranges hold tiles of the unit spanning global
// tiles [p0, p1), and the first of them (CTA of tile x: floor(((x+1)NC-1)/T)).
__device__ __forceinline__ int unit_segments(int p0, int p1, int T, int NC, int& c_lo, int& first_slot, int u) {
  if (p1 <= p0) return 0;
  c_lo = static_cast<int>((static_cast<int64_t>(p0 + 1) * NC - 1) / T);
  const int c_hi = static_cast<int>((static_cast<int64_t>(p1) * NC - 1) / T);
  first_slot = static_cast<int>(static_cast<int64_t>(c_lo) * T / NC) == p0 ? c_lo : NC + u;
  int n = 1;
  for (int c = c_lo + 1; c <= c_hi; ++c)
    if (static_cast<int64_t>(c) * T / NC < static_cast<int64_t>(c + 1) * T / NC) ++n;
  return n;
}

// Combine unit u = (b, j) from its segment partials (none for an empty unit):
// new-token join in score space, gate, fp32 store, write-back of the entry.
// All threads of the CTA take part; qs holds the unit's rotated q.
template <int D, int GP, bool PAGED>
__device__ void fused_combine(const FusedArgs& a, int u, const int* P, int T, const float* qs, float* sn) {
  const int Hkv = a.Hkv, G = a.G, Hq = Hkv * G, NC = a.ctas;
  const int b = u / Hkv, j = u - b * Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const CacheView& c = a.c;
  const uint16_t* kh = a.khat + static_cast<int64_t>(u) * D;
  // new-token scores (base 2), one warp per head
  for (int g = warp; g < G; g += kWarps) {
    float dot = 0.f;
    for (int d = lane; d < D; d += 32) dot = fmaf(qs[g * D + d], bf16_to_f32(kh[d]), dot);
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) dot += __shfl_xor_sync(kFull, dot, w);
    if (lane == 0) sn[g] = dot;
  }
  __syncthreads();
  int c_lo = 0, first_slot = 0;
  const int p0 = P[u], p1 = P[u + 1];
  const int nseg = unit_segments(p0, p1, T, NC, c_lo, first_slot, u);
  const int c_hi = p1 > p0 ? static_cast<int>((static_cast<int64_t>(p1) * NC - 1) / T) : c_lo - 1;
  const int stride = GP * (D + 2);
  (void)nseg;
  for (int e = threadIdx.x * 4; e < G * D; e += kThreads * 4) {
    const int g = e / D, d = e - g * D;
    const int h = j * G + g;
    float M = sn[g];
    for (int cc = c_lo; cc <= c_hi; ++cc) {
      const bool first = cc == c_lo;
      if (!first && !(static_cast<int64_t>(cc) * T / NC < static_cast<int64_t>(cc + 1) * T / NC)) continue;
      const float* pk = a.part + static_cast<int64_t>(first ? first_slot : cc) * stride;
      M = fmaxf(M, pk[GP * D + g]);
    }
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int cc = c_lo; cc <= c_hi; ++cc) {
      const bool first = cc == c_lo;
      if (!first && !(static_cast<int64_t>(cc) * T / NC < static_cast<int64_t>(cc + 1) * T / NC)) continue;
      const float* pk = a.part + static_cast<int64_t>(first ? first_slot : cc) * stride;
      const float w = exp2_fast(pk[GP * D + g] - M);
      L = fmaf(w, pk[GP * D + GP + g], L);
      const float4 v = *reinterpret_cast<const float4*>(pk + g * D + d);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    const float wn = exp2_fast(sn[g] - M);
    L += wn;
    const uint2 vw = *reinterpret_cast<const uint2*>(a.v_new + (static_cast<int64_t>(b) * Hkv + j) * D + d);
    acc.x = fmaf(wn, bf16_lo(vw.x), acc.x);
    acc.y = fmaf(wn, bf16_hi(vw.x), acc.y);
    acc.z = fmaf(wn, bf16_lo(vw.y), acc.z);
    acc.w = fmaf(wn, bf16_hi(vw.y), acc.w);
    float sig = 1.f;
    if (a.gate) sig = 1.f / (1.f + expf(-bf16_to_f32(a.gate[static_cast<int64_t>(b) * Hq + h])));
    const float scale = sig / L;
    *reinterpret_cast<float4*>(a.out + (static_cast<int64_t>(b) * Hq + h) * D + d) =
        make_float4(acc.x * scale, acc.y * scale, acc.z * scale, acc.w * scale);
  }
  // write-back of the new entry: every segment of this unit has finished reading
  if (a.write_back) {
    int64_t wb = -1;
    if constexpr (PAGED) {
      const int n = min(max(c.seq_len[b], 0), min(a.max_len, c.bt_stride * c.P));
      const int pi = n / c.P;
      const int pg = pi < c.bt_stride ? c.block_table[static_cast<int64_t>(b) * c.bt_stride + pi] : -1;
      if (pg >= 0 && pg < c.n_rows)
        wb = ((static_cast<int64_t>(pg) * Hkv + j) * c.P + n % c.P) * D;
      else if (threadIdx.x == 0)
        raise_error(a.err, ERR_INDEX);
    } else {
      const int row = c.stream_rows ? c.stream_rows[b] : b;
      const int head = c.ring_head[b], cnt = c.ring_count[b];
      if (!(row < 0 || row >= c.n_rows || head < 0 || head >= c.R || cnt < 0 || cnt > c.R))
        wb = ((static_cast<int64_t>(row) * Hkv + j) * c.R + head) * D;
    }
    if (wb >= 0) {
      const uint16_t* vn = a.v_new + (static_cast<int64_t>(b) * Hkv + j) * D;
      for (int d = threadIdx.x * 4; d < D; d += kThreads * 4) {
        *reinterpret_cast<uint2*>(c.k + wb + d) = *reinterpret_cast<const uint2*>(kh + d);
        *reinterpret_cast<uint2*>(c.v + wb + d) = *reinterpret_cast<const uint2*>(vn + d);
      }
    }
  }
  if (threadIdx.x == 0) a.counters[u] = 0;
  __syncthreads();
}

template <int D, int GP, bool PAGED>
__global__ void __launch_bounds__(kThreads, 2) decode_fused_kernel(const FusedArgs a) {
  using Gm = Geo<D, GP>;
  using F = FGeo<D, GP>;
  constexpr int LPK = Gm::LPK, KPS = Gm::KPS, J = Gm::J, KT = Gm::KT, SK = Gm::SK;
  constexpr int SUB = Gm::SUB, NS = Gm::NS;
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const CacheView& c = a.c;
  const int Hkv = a.Hkv, U = a.B * Hkv, G = a.G;
  const int NC = gridDim.x, cta = blockIdx.x;
  int* P = reinterpret_cast<int*>(smem + F::TAB_OFF);  // [U + 1] tile prefix over units
  int* N = P + U + 1;                                   // [U] cached keys per unit
  float* qs = reinterpret_cast<float*>(smem + F::QS_OFF);
  float* sn = reinterpret_cast<float*>(smem + F::SN_OFF);
  int* flag = reinterpret_cast<int*>(smem + F::FLAG_OFF);

  // ---- unit table from caller metadata
  for (int u = threadIdx.x; u < U; u += kThreads) {
    const int b = u / Hkv;
    const int n = unit_length<PAGED>(c, b, a.max_len, cta == 0 && u - b * Hkv == 0, a.err);
    N[u] = n;
    P[u + 1] = (n + SK - 1) / SK;
  }
  if (threadIdx.x == 0) P[0] = 0;
  __syncthreads();
  block_scan_inclusive<kThreads>(P + 1, U);
  const int T = P[U];
  const int g0 = static_cast<int>(static_cast<int64_t>(cta) * T / NC);
  const int g1 = static_cast<int>(static_cast<int64_t>(cta + 1) * T / NC);
  const int span = g1 - g0;
  const int my_n = span > warp ? (span - warp + kWarps - 1) / kWarps : 0;
  uint8_t* wsm = smem + warp * NS * Gm::STAGE;
  const uint32_t bar0 = smem_addr(smem + Gm::BAR_OFF) + warp * NS * 8;
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();

  // The previous call may still be writing the cache (its new entries) and
  // reading the workspace: everything below waits for it.
  pdl_wait();
  pdl_trigger();

  const uint64_t policy = l2_evict_first_policy();
  int u_iss = my_n > 0 ? unit_of(P, U, g0 + warp) : 0;
  auto issue = [&](int it) {
    const int g = g0 + warp + kWarps * it;
    while (P[u_iss + 1] <= g) ++u_iss;
    const int u = u_iss;
    const int b = u / Hkv, j = u - b * Hkv;
    const int k0 = (g - P[u]) * SK;
    const int cnt = min(SK, N[u] - k0);
    const uint32_t bar = bar0 + 8 * (it % NS);
    const uint32_t kd = smem_addr(wsm + (it % NS) * Gm::STAGE);
    const uint32_t vd = kd + Gm::TILE;
    mbar_arrive_expect_tx(bar, 2u * cnt * Gm::ROW);
    if constexpr (PAGED) {
      const int32_t* bt = c.block_table + static_cast<int64_t>(b) * c.bt_stride;
      int t = k0, done = 0;
      while (t < k0 + cnt) {
        const int pi = t / c.P;
        const int off = t - pi * c.P;
        int pg = bt[pi];
        if (pg < 0 || pg >= c.n_rows) {
          raise_error(a.err, ERR_INDEX);
          pg = 0;
        }
        const int run = min(c.P - off, k0 + cnt - t);
        const int64_t src = ((static_cast<int64_t>(pg) * Hkv + j) * c.P + off) * D;
        bulk_copy_g2s(kd + done * Gm::ROW, c.k + src, run * Gm::ROW, bar, policy);
        bulk_copy_g2s(vd + done * Gm::ROW, c.v + src, run * Gm::ROW, bar, policy);
        t += run;
        done += run;
      }
    } else {
      const int row = c.stream_rows ? c.stream_rows[b] : b;
      const int n = N[u];
      const int head = c.ring_head[b];
      const int start = head - n < 0 ? head - n + c.R : head - n;
      const int64_t base = (static_cast<int64_t>(row) * Hkv + j) * c.R * D;
      int phys = start + k0;
      if (phys >= c.R) phys -= c.R;
      const int run1 = min(cnt, c.R - phys);
      bulk_copy_g2s(kd, c.k + base + static_cast<int64_t>(phys) * D, run1 * Gm::ROW, bar, policy);
      bulk_copy_g2s(vd, c.v + base + static_cast<int64_t>(phys) * D, run1 * Gm::ROW, bar, policy);
      if (run1 < cnt) {
        bulk_copy_g2s(kd + run1 * Gm::ROW, c.k + base, (cnt - run1) * Gm::ROW, bar, policy);
        bulk_copy_g2s(vd + run1 * Gm::ROW, c.v + base, (cnt - run1) * Gm::ROW, bar, policy);
      }
    }
  };
  if (lane == 0) {
    const int pre = my_n < NS ? my_n : NS;
    for (int it = 0; it < pre; ++it) issue(it);
  }

  float* ML = reinterpret_cast<float*>(smem + Gm::ML_OFF);
  int* SLOT = reinterpret_cast<int*>(smem + Gm::SLOT_OFF);
  float* psm = reinterpret_cast<float*>(smem + Gm::PSM_OFF) + warp * (32 + GP);
  const int dl = (lane % LPK) * 8;
  const int half = lane / LPK;
  const int key_s = ((lane % LPK) / GP) * KPS + half;

  bool failed = false;
  int it = 0;
  int deferred = -1;
  bool first_seg = true;
  for (int u = span > 0 ? unit_of(P, U, g0) : U; u < U && P[u] < g1; ++u) {
    if (P[u + 1] == P[u]) continue;  // a unit with no cached keys
    const int ge = min(g1, P[u + 1]);
    const int b = u / Hkv, j = u - b * Hkv;

    // the unit's rotated q; the CTA holding the unit's first tile also writes
    // the unit's K entry (read by whichever CTA combines the unit)
    fused_rope_q<D, GP>(a, b, j, qs);
    if (P[u] >= g0) fused_k_entry<D>(a, b, j, a.khat + static_cast<int64_t>(u) * D);
    __syncthreads();
    // packed fp32 pairs: the FMAs below are Blackwell's two-wide FFMA2
    float2 q2[GP][4];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      const float4 x0 = *reinterpret_cast<const float4*>(qs + g * D + dl);
      const float4 x1 = *reinterpret_cast<const float4*>(qs + g * D + dl + 4);
      q2[g][0] = make_float2(x0.x, x0.y); q2[g][1] = make_float2(x0.z, x0.w);
      q2[g][2] = make_float2(x1.x, x1.y); q2[g][3] = make_float2(x1.z, x1.w);
    }
    float2 o2[GP][4];
#pragma unroll
    for (int g = 0; g < GP; ++g)
#pragma unroll
      for (int e = 0; e < 4; ++e) o2[g][e] = make_float2(0.f, 0.f);
    float m_run = -INFINITY, l_run = 0.f;
    int last_stage = -1;

    for (;;) {
      const int g = g0 + warp + kWarps * it;
      if (it >= my_n || g >= ge) break;
      const int stg = it % NS;
      if (!failed) {
        const bool ok = __all_sync(kFull, mbar_wait_bounded(bar0 + 8 * stg, (it / NS) & 1));
        if (!ok) {
          failed = true;
          if (lane == 0) raise_error(a.err, ERR_TIMEOUT);
        }
      }
      if (!failed) {
        const int nstage = min(SK, N[u] - (g - P[u]) * SK);
#pragma unroll 1
        for (int sb = 0; sb < SUB; ++sb) {
          const int nvalid = nstage - sb * KT;
          if (nvalid <= 0) break;
          const uint4* Ks = reinterpret_cast<const uint4*>(wsm + stg * Gm::STAGE) + sb * (KT * D / 8);
          const uint4* Vs = Ks + Gm::TILE / 16;
          float sp[J * GP];
#pragma unroll
          for (int jj = 0; jj < J; ++jj) {
            float2 k2[4];
            unpack8x2(Ks[jj * 32 + lane], k2);
#pragma unroll
            for (int h = 0; h < GP; ++h) {
              float2 a2 = __fmul2_rn(q2[h][0], k2[0]);
              a2 = __ffma2_rn(q2[h][1], k2[1], a2);
              a2 = __ffma2_rn(q2[h][2], k2[2], a2);
              a2 = __ffma2_rn(q2[h][3], k2[3], a2);
              sp[jj * GP + h] = a2.x + a2.y;
            }
          }
          float s = transpose_reduce<LPK>(sp, lane);
          if (key_s >= nvalid) s = -INFINITY;
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
          // rescale only when some head's running maximum moved
          if (__any_sync(kFull, corr != 1.f)) {
#pragma unroll
            for (int h = 0; h < GP; ++h) {
              const float cr = psm[32 + h];
              const float2 c2 = make_float2(cr, cr);
#pragma unroll
              for (int e = 0; e < 4; ++e) o2[h][e] = __fmul2_rn(o2[h][e], c2);
            }
          }
          if (nvalid >= KT) {
#pragma unroll
            for (int jj = 0; jj < J; ++jj) {
              float2 v2[4];
              unpack8x2(Vs[jj * 32 + lane], v2);
              const float* pp = psm + half * LPK + jj * GP;
#pragma unroll
              for (int h = 0; h < GP; ++h) {
                const float2 p2 = make_float2(pp[h], pp[h]);
#pragma unroll
                for (int e = 0; e < 4; ++e) o2[h][e] = __ffma2_rn(p2, v2[e], o2[h][e]);
              }
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < J; ++jj) {
              if (jj * KPS + half < nvalid) {
                float2 v2[4];
                unpack8x2(Vs[jj * 32 + lane], v2);
                const float* pp = psm + half * LPK + jj * GP;
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                  const float2 p2 = make_float2(pp[h], pp[h]);
#pragma unroll
                  for (int e = 0; e < 4; ++e) o2[h][e] = __ffma2_rn(p2, v2[e], o2[h][e]);
                }
              }
            }
          }
          __syncwarp();
        }
      }
      last_stage = stg;
      if (it + NS < my_n) {
        if (g + kWarps >= ge) {
          deferred = it + NS;
        } else if (lane == 0 && !failed) {
          fence_proxy_async_smem();
          issue(it + NS);
        }
      }
      ++it;
    }

    // ---- merge the warps' states for this segment into its partial slot
#pragma unroll
    for (int w = GP; w < 32; w <<= 1) l_run += __shfl_xor_sync(kFull, l_run, w);
#pragma unroll
    for (int w = LPK; w < 32; w <<= 1)
#pragma unroll
      for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          o2[h][e].x += __shfl_xor_sync(kFull, o2[h][e].x, w);
          o2[h][e].y += __shfl_xor_sync(kFull, o2[h][e].y, w);
        }
    if (last_stage >= 0 && lane < LPK) {
      float* os = reinterpret_cast<float*>(wsm + last_stage * Gm::STAGE);
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        *reinterpret_cast<float4*>(os + h * D + dl) = make_float4(o2[h][0].x, o2[h][0].y, o2[h][1].x, o2[h][1].y);
        *reinterpret_cast<float4*>(os + h * D + dl + 4) = make_float4(o2[h][2].x, o2[h][2].y, o2[h][3].x, o2[h][3].y);
      }
    }
    if (lane < GP) {
      ML[warp * 2 * GP + lane] = last_stage >= 0 ? m_run : -INFINITY;
      ML[warp * 2 * GP + GP + lane] = last_stage >= 0 ? l_run : 0.f;
    }
    if (lane == 0) SLOT[warp] = last_stage;
    __syncthreads();
    const int slot = first_seg ? cta : NC + u;
    float* dst = a.part + static_cast<int64_t>(slot) * (GP * (D + 2));
    for (int e = threadIdx.x; e < GP * D; e += kThreads) {
      const int h = e / D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ML[w * 2 * GP + h]);
      float acc = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const int st = SLOT[w];
          if (st >= 0) {
            const float* os = reinterpret_cast<const float*>(smem + (w * NS + st) * Gm::STAGE);
            acc = fmaf(exp2_fast(ML[w * 2 * GP + h] - M), os[e], acc);
          }
        }
      }
      dst[e] = acc;
    }
    if (threadIdx.x < GP) {
      const int h = threadIdx.x;
      float M = -INFINITY;
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ML[w * 2 * GP + h]);
      float L = 0.f;
      if (M != -INFINITY)
        for (int w = 0; w < kWarps; ++w) L = fmaf(exp2_fast(ML[w * 2 * GP + h] - M), ML[w * 2 * GP + GP + h], L);
      dst[GP * D + h] = M;
      dst[GP * D + GP + h] = L;
    }
    // count this segment; the CTA finishing the unit's last segment combines it
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      int c_lo = 0, fs = 0;
      const int nseg = unit_segments(P[u], P[u + 1], T, NC, c_lo, fs, u);
      *flag = atomicAdd(a.counters + u, 1) == nseg - 1;
    }
    __syncthreads();
    if (deferred >= 0) {
      if (lane == 0 && !failed) {
        fence_proxy_async_smem();
        issue(deferred);
      }
      deferred = -1;
    }
    if (*flag) {
      __threadfence();
      fused_combine<D, GP, PAGED>(a, u, P, T, qs, sn);
    }
    first_seg = false;
  }

  // units with no cached keys have no segments: CTA u % NC combines them
  for (int u = cta; u < U; u += NC) {
    if (N[u] != 0) continue;
    const int b = u / Hkv, j = u - b * Hkv;
    fused_rope_q<D, GP>(a, b, j, qs);
    fused_k_entry<D>(a, b, j, a.khat + static_cast<int64_t>(u) * D);
    __threadfence();
    __syncthreads();
    fused_combine<D, GP, PAGED>(a, u, P, T, qs, sn);
  }
}

template <int D, int GP, bool PAGED>
cudaError_t fused_launch(const FusedArgs& a, cudaStream_t s) {
  using F = FGeo<D, GP>;
  auto k = decode_fused_kernel<D, GP, PAGED>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, F::SMEM_MAX);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const size_t smem = F::TAB_OFF + (2 * a.B * a.Hkv + 1) * sizeof(int);
  return launch_pdl(k, dim3(a.ctas), dim3(kThreads), smem, s, a);
}

template <int D, int GP>
cudaError_t fused_dispatch(const FusedArgs& a, cudaStream_t s) {
  return a.c.paged ? fused_launch<D, GP, true>(a, s) : fused_launch<D, GP, false>(a, s);
}

template <int D, int GP, bool PAGED>
cudaError_t split_launch(const SplitArgs& a, int G, cudaStream_t s) {
  using Gm = Geo<D, GP>;
  auto k = decode_split_kernel<D, GP, PAGED>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM_MAX);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const size_t smem = Gm::TAB_OFF + (2 * a.B * a.Hkv + 1) * sizeof(int);
  return launch_pdl(k, dim3(a.ctas), dim3(kThreads), smem, s, a, G);
}

template <int D, int GP>
cudaError_t split_dispatch_paged(const SplitArgs& a, int G, cudaStream_t s) {
  return a.c.paged ? split_launch<D, GP, true>(a, G, s) : split_launch<D, GP, false>(a, G, s);
}

int padded_group(int G) { return G <= 2 ? 2 : (G <= 4 ? 4 : (G <= 8 ? 8 : 0)); }

template <int D>
int geo_smem_max(int GP) {
  return GP == 2 ? Geo<D, 2>::SMEM_MAX : GP == 4 ? Geo<D, 4>::SMEM_MAX : GP == 8 ? Geo<D, 8>::SMEM_MAX : 0;
}
template <int D>
int geo_stage_keys(int GP) {
  return GP == 2 ? Geo<D, 2>::SK : GP == 4 ? Geo<D, 4>::SK : GP == 8 ? Geo<D, 8>::SK : 0;
}

}  // namespace

cudaError_t launch_decode_split(const SplitArgs& a, int D, int G, cudaStream_t s) {
  const int GP = padded_group(G);
  if (a.B * a.Hkv > kMaxUnits) return cudaErrorNotSupported;
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
  if (GP == 0) return 0;
  return D == 256 ? geo_stage_keys<256>(GP) : D == 128 ? geo_stage_keys<128>(GP) : 0;
}

int decode_split_ctas_per_sm(int D, int G) {
  const int GP = padded_group(G);
  const int smem = GP == 0 ? 0 : D == 256 ? geo_smem_max<256>(GP) : D == 128 ? geo_smem_max<128>(GP) : 0;
  if (smem == 0) return 0;
  // 228 KB of shared memory per SM, 1 KB of it reserved per resident CTA
  const int per_sm = 233472 / (smem + 1024);
  return per_sm > 2 ? 2 : per_sm;
}

int decode_max_units() { return kMaxUnits; }

cudaError_t launch_decode_fused(const FusedArgs& a, int D, cudaStream_t s) {
  const int GP = padded_group(a.G);
  if (a.B * a.Hkv > kMaxUnits) return cudaErrorNotSupported;
  if (D == 256) {
    if (GP == 2) return fused_dispatch<256, 2>(a, s);
    if (GP == 4) return fused_dispatch<256, 4>(a, s);
    if (GP == 8) return fused_dispatch<256, 8>(a, s);
  } else if (D == 128) {
    if (GP == 2) return fused_dispatch<128, 2>(a, s);
    if (GP == 4) return fused_dispatch<128, 4>(a, s);
    if (GP == 8) return fused_dispatch<128, 8>(a, s);
  }
  return cudaErrorNotSupported;
}

int decode_fused_ctas_per_sm(int D, int G) {
  const int GP = padded_group(G);
  int smem = 0;
  if (D == 256) smem = GP == 2 ? FGeo<256, 2>::SMEM_MAX : GP == 4 ? FGeo<256, 4>::SMEM_MAX : GP == 8 ? FGeo<256, 8>::SMEM_MAX : 0;
  if (D == 128) smem = GP == 2 ? FGeo<128, 2>::SMEM_MAX : GP == 4 ? FGeo<128, 4>::SMEM_MAX : GP == 8 ? FGeo<128, 8>::SMEM_MAX : 0;
  if (smem == 0) return 0;
  // 228 KB of shared memory per SM; 1 KB reserved and the static block-scan scratch per CTA
  const int per_sm = 233472 / (smem + 1024 + 64);
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
  int p2 = 1;
  while (p2 < dsplit) p2 <<= 1;
  dsplit = p2 > dmax ? dmax : p2;
  const int tph = D / 4 / dsplit;
  const int threads = (G * tph + 31) / 32 * 32;
  dim3 grid(dsplit, a.Hkv, a.B);
  dim3 block(threads);
  const size_t smem = static_cast<size_t>(threads / tph) * a.split_ctas * sizeof(float);
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
