// Decode attention: the split-K pass over the cached keys and the LSE combine
// that joins the new token in score space.
//
// Method ("vllm-omni commits", score-space join commit): the cached keys (n of
// them) and the new key are scored separately and their score vectors meet in
// one softmax; nothing cache-sized is copied, and the new K/V entry is written
// into its slot afterwards. A ring's slots need no reordering (softmax is
// order-free, cached keys carry their own rotary phase); unwritten slots are
// masked. Grouped-query attention shares each KV head's loads among its G
// query heads ("vllm-omni commits", talker export commit). Splitting the keys
// over many CTAs and merging their partial softmax states follows "TensorFold
// PR #608" (the split "shared" kernel plus a merge, the lessons that the grid
// must fill the GPU and that a merge must not be a chain of dependent loads).
//
// GB300 design.
//  * Work split (stream-K). A "unit" is one (stream, KV head). Its cached keys
//    are visited in groups of 16 rows: 16-row runs of a page (a page of P
//    rows gives ceil(P / 16) groups), or 16-slot blocks of the ring's physical
//    slots (only the blocks that hold valid slots; softmax does not care about
//    the order). A stage tile is 256 / D groups (16 KB of K and V). All units'
//    tiles are laid end to end and the grid - one CTA per SM - cuts that
//    sequence into equal contiguous ranges, so every CTA moves the same number
//    of bytes whatever the mix of lengths. Each piece of a unit inside one CTA
//    (a "segment") leaves one partial softmax state (m, l, o); the combine
//    merges a unit's segments.
//  * Loads. Each warp owns a ring of NS stage buffers. One lane issues 2D
//    tensor TMA copies (boxes of 16 rows x 64 bf16, 128-byte swizzle; one box
//    per 64 dims of K and of V per group) for the warp's tile NS ahead, with
//    completion counted in bytes on the stage's mbarrier; the ring keeps
//    streaming across segment boundaries. Rows a box brings in that are not
//    valid keys (past a unit's length, past a page, outside a ring's valid
//    slots, or zero-filled past the pool) are masked: their scores are set to
//    -inf and their V rows are zeroed in shared memory before use.
//  * Math on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate).
//    The KV stream is HBM-bound at G flops per byte; the tensor cores are used
//    because they cut the instructions per byte about tenfold against fp32
//    FMAs, which otherwise limit the issue rate. Per group of 16 keys:
//      S^T (16 keys x 8 cols) = K (16 x D) . Q^T (D x 8 cols)
//      O^T (D x 8 cols)      += V^T (D x 16) . P^T (16 x 8 cols)
//    The 8 (or 2 x 8) columns hold each query head twice: once as the bf16
//    rounding of the pre-scaled rotated q, once as the bf16 rounding of what
//    is left ("hi" and "lo"), so q keeps 16 significant bits; the two score
//    columns of a head are added. The probabilities are split into hi and lo
//    bf16 parts the same way, so the value sum sees 16-bit probabilities; the
//    two output columns of a head are added at the end. K and V enter the
//    tensor cores exactly (they are bf16). The score fragment turns into the
//    PV operand in registers (movmatrix transposes); online softmax in base 2
//    runs on the score fragment, and the output is rescaled only when some
//    head's running maximum moved.
#include "common.cuh"
#include "mma.cuh"

namespace dattn {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxUnits = 1024;   // (stream, KV head) units per call
constexpr int kGroup = 16;        // keys per MMA group
constexpr int kBoxBytes = kGroup * 128;  // one TMA box: 16 rows x 64 bf16

template <int D, int NT>
struct Geo {
  static constexpr int GP = 4 * NT;                  // heads per partial slot
  static constexpr int KSTEPS = D / 16;              // MMA k-steps of a score, m-tiles of an output
  static constexpr int BOXES = D / 64;               // TMA boxes per 16-row group of K (or V)
  static constexpr int GBYTES = BOXES * kBoxBytes;   // K (or V) bytes of one group
  static constexpr int KG = 256 / D;                 // groups per stage tile
  static constexpr int KHALF = KG * GBYTES;          // K part of a stage; V follows
  static constexpr int STAGE = 2 * KHALF;
  static constexpr int NS = 3;
  static constexpr int BAR_OFF = kWarps * NS * STAGE;        // from the 1024-aligned base
  static constexpr int ML_OFF = BAR_OFF + kWarps * NS * 8;   // float [kWarps][2*GP]
  static constexpr int SLOT_OFF = ML_OFF + kWarps * 2 * GP * 4;  // int [kWarps]
  static constexpr int TAB_OFF = (SLOT_OFF + kWarps * 4 + 15) / 16 * 16;
  static constexpr int SMEM_MAX = 1024 + TAB_OFF + (2 * kMaxUnits + 1) * 4;
  static_assert(D == 128 || D == 256, "head_dim");
  static_assert(GP * D * 4 <= STAGE, "a stage buffer holds one warp's partial output");
};

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

// First 16-slot block of a ring holding `n` valid slots before `head`.
__device__ __forceinline__ int ring_first_block(int head, int n, int R) {
  const int start = head - n < 0 ? head - n + R : head - n;
  return start >> 4;
}

// 16-row groups of a unit with n cached keys.
template <bool PAGED>
__device__ __forceinline__ int unit_groups(const CacheView& c, int b, int n) {
  if (n <= 0) return 0;
  if constexpr (PAGED) {
    const int gpp = (c.P + kGroup - 1) / kGroup;
    const int full = n / c.P, rest = n - full * c.P;
    return full * gpp + (rest + kGroup - 1) / kGroup;
  } else {
    const int R = c.R, nb = (R + kGroup - 1) / kGroup;
    if (n >= R) return nb;
    const int head = c.ring_head[b];
    const int start = head - n < 0 ? head - n + R : head - n;
    const int b0 = start >> 4, end = start + n - 1;
    if (end < R) return (end >> 4) - b0 + 1;
    return min(nb, nb - b0 + ((end - R) >> 4) + 1);  // wraps past the last slot
  }
}

template <int D, int NT, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1) decode_split_kernel(const __grid_constant__ SplitArgs a, int G) {
  using Gm = Geo<D, NT>;
  constexpr int GP = Gm::GP, KSTEPS = Gm::KSTEPS, BOXES = Gm::BOXES, KG = Gm::KG, NS = Gm::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
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
    P[u + 1] = (unit_groups<PAGED>(c, b, n) + KG - 1) / KG;
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
  const uint32_t wsm_a = smem_addr(wsm);
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
    const int n = N[u];
    const int gb = (g - P[u]) * KG;
    const int gn = min(KG, unit_groups<PAGED>(c, b, n) - gb);
    const uint32_t bar = bar0 + 8 * (it % NS);
    const uint32_t kd = wsm_a + (it % NS) * Gm::STAGE;
    mbar_arrive_expect_tx(bar, 2u * gn * Gm::GBYTES);
    for (int kg = 0; kg < gn; ++kg) {
      const int gi = gb + kg;
      int row0;
      if constexpr (PAGED) {
        const int gpp = (c.P + kGroup - 1) / kGroup;
        const int pi = gi / gpp;
        int pg = c.block_table[static_cast<int64_t>(b) * c.bt_stride + pi];
        if (pg < 0 || pg >= c.n_rows) {
          raise_error(a.err, ERR_INDEX);
          pg = 0;
        }
        row0 = (pg * Hkv + j) * c.P + (gi - pi * gpp) * kGroup;
      } else {
        const int nb = (c.R + kGroup - 1) / kGroup;
        int pb = ring_first_block(c.ring_head[b], n, c.R) + gi;
        if (pb >= nb) pb -= nb;
        const int row = c.stream_rows ? c.stream_rows[b] : b;
        row0 = (row * Hkv + j) * c.R + pb * kGroup;
      }
#pragma unroll
      for (int x = 0; x < BOXES; ++x) {
        tma_load_2d(kd + kg * Gm::GBYTES + x * kBoxBytes, &a.tmap_k, 64 * x, row0, bar, policy);
        tma_load_2d(kd + Gm::KHALF + kg * Gm::GBYTES + x * kBoxBytes, &a.tmap_v, 64 * x, row0, bar,
                    policy);
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

  // Per-lane ldmatrix offsets inside a group's 2 KB boxes (128-byte swizzle:
  // the 16-byte chunk index is XORed with the row mod 8). K (scores, A = K):
  // matrix m = lane / 8 covers rows 8 * (m & 1) + 0..7 and chunk (m >> 1) of
  // a k-step's pair of chunks. V (outputs, A = V^T, loaded transposed):
  // matrix m covers rows 8 * (m >> 1) + 0..7 and chunk (m & 1).
  const int lr = lane & 7, lm = lane >> 3;
  uint32_t koff[4], voff[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int rk = lr + 8 * (lm & 1), rv = lr + 8 * (lm >> 1);
    koff[q] = rk * 128 + (((2 * q + (lm >> 1)) ^ lr) << 4);
    voff[q] = rv * 128 + (((2 * q + (lm & 1)) ^ lr) << 4);
  }
  const int fg = lane >> 2, fc = 2 * (lane & 3);  // fragment row group, column pair
  // heads of this lane's score / output columns (e = 0, 1): hi/lo columns of
  // one head are lanes l and l ^ 2 (NT == 1) or tiles 0 and 1 (NT == 2)
  const int hbase = NT == 1 ? 2 * (lane & 1) : fc;
  const bool lo_lane = NT == 1 && (lane & 2) != 0;

  bool failed = false;
  int it = 0;
  int deferred = -1;
  bool first_seg = true;
  for (int u = span > 0 ? unit_of(P, U, g0) : U; u < U && P[u] < g1; ++u) {
    if (P[u + 1] == P[u]) continue;  // a unit with no cached keys
    const int ge = min(g1, P[u + 1]);
    const int b = u / Hkv, j = u - b * Hkv;
    const int n = N[u];

    // q^T as B fragments: column n = fg of tile t holds head (hi or lo part)
    uint32_t qb[KSTEPS][NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int head = NT == 1 ? (fg & 3) : fg;
      const bool lo = NT == 1 ? fg >= 4 : t == 1;
      const float* src = a.qhat + (static_cast<int64_t>(b) * Hkv * G + j * G + head) * D + fc;
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          float2 x = make_float2(0.f, 0.f);
          if (head < G) x = *reinterpret_cast<const float2*>(src + ks * 16 + h2 * 8);
          uint32_t hi, lw;
          split_bf16x2(x.x, x.y, hi, lw);
          qb[ks][t][h2] = lo ? lw : hi;
        }
      }
    }
    float o[KSTEPS][NT][4];
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt)
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][t][e] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    int last_stage = -1;
    const int ngroups = unit_groups<PAGED>(c, b, n);
    int ring_b0 = 0;
    if constexpr (!PAGED) ring_b0 = ring_first_block(c.ring_head[b], n, c.R);

    for (;;) {
      const int g = g0 + warp + kWarps * it;
      if (it >= my_n || g >= ge) break;
      const int stg = it % NS;
      if (!failed) {
        // the whole warp agrees on the outcome, so the collectives below stay converged
        const bool ok = __all_sync(kFull, mbar_wait_bounded(bar0 + 8 * stg, (it / NS) & 1));
        if (!ok) {
          failed = true;
          if (lane == 0) raise_error(a.err, ERR_TIMEOUT);
        }
      }
      if (!failed) {
        const int gb = (g - P[u]) * KG;
        const int gn = min(KG, ngroups - gb);
#pragma unroll 1
        for (int kg = 0; kg < gn; ++kg) {
          const uint32_t kbase = wsm_a + stg * Gm::STAGE + kg * Gm::GBYTES;
          const uint32_t vbase = kbase + Gm::KHALF;
          // ---- which of the group's 16 rows are valid keys
          const int gi = gb + kg;
          const int r = lane & 15;
          bool valid;
          if constexpr (PAGED) {
            const int gpp = (c.P + kGroup - 1) / kGroup;
            const int pi = gi / gpp, off = (gi - pi * gpp) * kGroup + r;
            valid = off < c.P && pi * c.P + off < n;
          } else {
            const int nb = (c.R + kGroup - 1) / kGroup;
            int pb = ring_b0 + gi;
            if (pb >= nb) pb -= nb;
            const int slot = pb * kGroup + r;
            int d = c.ring_head[b] - 1 - slot;
            if (d < 0) d += c.R;
            valid = slot < c.R && d < n;
          }
          const uint32_t mask = __ballot_sync(kFull, valid) & 0xffffu;
          if (mask != 0xffffu) {
            // zero the V rows of invalid keys (their probabilities are 0, but
            // the rows may hold NaN and 0 * NaN is NaN)
            uint8_t* vg = wsm + stg * Gm::STAGE + Gm::KHALF + kg * Gm::GBYTES;
            for (int i = lane; i < kGroup * BOXES * 8; i += 32) {
              const int row = i / (BOXES * 8), rest = i - row * (BOXES * 8);
              if (!((mask >> row) & 1u))
                *reinterpret_cast<uint4*>(vg + (rest >> 3) * kBoxBytes + row * 128 + (rest & 7) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();  // before the stage is refilled by TMA
            __syncwarp();
          }

          // ---- scores S^T = K . Q^T (two accumulator chains)
          float sacc[2][NT][4];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
              for (int e = 0; e < 4; ++e) sacc[h2][t][e] = 0.f;
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            uint32_t af[4];
            ldsm_x4(kbase + (ks >> 2) * kBoxBytes + koff[ks & 3], af);
#pragma unroll
            for (int t = 0; t < NT; ++t) mma_bf16(sacc[ks & 1][t], af, qb[ks][t][0], qb[ks][t][1]);
          }
          // full scores of heads hbase + e at keys fg (i = e) and fg + 8 (i = 2 + e)
          float s[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (NT == 1) {
              const float x = sacc[0][0][i] + sacc[1][0][i];
              s[i] = x + __shfl_xor_sync(kFull, x, 2);
            } else {
              s[i] = (sacc[0][0][i] + sacc[1][0][i]) + (sacc[0][NT - 1][i] + sacc[1][NT - 1][i]);
            }
          }
          if (!((mask >> fg) & 1u)) s[0] = s[1] = -INFINITY;
          if (!((mask >> (fg + 8)) & 1u)) s[2] = s[3] = -INFINITY;

          // ---- online softmax (base 2), per head over the 16 keys
          float corr[2], p[4];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float mx = fmaxf(s[e], s[2 + e]);
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
            const float m_new = fmaxf(m_run[e], mx);
            const float ms = m_new == -INFINITY ? 0.f : m_new;
            corr[e] = exp2_fast(m_run[e] - ms);
            p[e] = exp2_fast(s[e] - ms);
            p[2 + e] = exp2_fast(s[2 + e] - ms);
            l_run[e] = fmaf(l_run[e], corr[e], p[e] + p[2 + e]);
            m_run[e] = m_new;
          }
          if (__any_sync(kFull, corr[0] != 1.f || corr[1] != 1.f)) {
#pragma unroll
            for (int mt = 0; mt < KSTEPS; ++mt)
#pragma unroll
              for (int t = 0; t < NT; ++t) {
                o[mt][t][0] *= corr[0];
                o[mt][t][1] *= corr[1];
                o[mt][t][2] *= corr[0];
                o[mt][t][3] *= corr[1];
              }
          }

          // ---- P^T as B fragments (hi and lo bf16 parts), via 8x8 transposes
          uint32_t pb[NT][2];
          {
            uint32_t h01, l01, h23, l23;
            split_bf16x2(p[0], p[1], h01, l01);
            split_bf16x2(p[2], p[3], h23, l23);
            if (NT == 1) {
              pb[0][0] = movm_t(lo_lane ? l01 : h01);
              pb[0][1] = movm_t(lo_lane ? l23 : h23);
            } else {
              pb[0][0] = movm_t(h01);
              pb[0][1] = movm_t(h23);
              pb[NT - 1][0] = movm_t(l01);
              pb[NT - 1][1] = movm_t(l23);
            }
          }

          // ---- outputs O^T += V^T . P^T
#pragma unroll
          for (int mt = 0; mt < KSTEPS; ++mt) {
            uint32_t af[4];
            ldsm_x4_t(vbase + (mt >> 2) * kBoxBytes + voff[mt & 3], af);
#pragma unroll
            for (int t = 0; t < NT; ++t) mma_bf16(o[mt][t], af, pb[t][0], pb[t][1]);
          }
        }
        __syncwarp();
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

    // ---- this warp's state: l summed over the lanes of a head, O^T to the
    // merge buffer as o[head][dim] (hi + lo columns)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      l_run[e] += __shfl_xor_sync(kFull, l_run[e], 4);
      l_run[e] += __shfl_xor_sync(kFull, l_run[e], 8);
      l_run[e] += __shfl_xor_sync(kFull, l_run[e], 16);
    }
    if (last_stage >= 0) {
      float* os = reinterpret_cast<float*>(wsm + last_stage * Gm::STAGE);
      const bool writer = NT == 2 || !lo_lane;
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float v;
          if (NT == 1) {
            v = o[mt][0][i] + __shfl_xor_sync(kFull, o[mt][0][i], 2);
          } else {
            v = o[mt][0][i] + o[mt][NT - 1][i];
          }
          if (writer) os[(hbase + (i & 1)) * D + mt * 16 + fg + 8 * (i >> 1)] = v;
        }
      fence_proxy_async_smem();  // the buffer is refilled by TMA after the merge
    }
    if (fg == 0 && (NT == 2 || !lo_lane)) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        ML[warp * 2 * GP + hbase + e] = last_stage >= 0 ? m_run[e] : -INFINITY;
        ML[warp * 2 * GP + GP + hbase + e] = last_stage >= 0 ? l_run[e] : 0.f;
      }
    }
    if (lane == 0) SLOT[warp] = last_stage;
    __syncthreads();
    // ---- merge the warps' states for this segment into its partial slot
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

// ---------------------------------------------------------------- launch

template <int D, int NT, bool PAGED>
cudaError_t split_launch(const SplitArgs& a, int G, cudaStream_t s) {
  using Gm = Geo<D, NT>;
  auto k = decode_split_kernel<D, NT, PAGED>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM_MAX);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const size_t smem = 1024 + Gm::TAB_OFF + (2 * a.B * a.Hkv + 1) * sizeof(int);
  return launch_pdl(k, dim3(a.ctas), dim3(kThreads), smem, s, a, G);
}

template <int D, int NT>
cudaError_t split_dispatch_paged(const SplitArgs& a, int G, cudaStream_t s) {
  return a.c.paged ? split_launch<D, NT, true>(a, G, s) : split_launch<D, NT, false>(a, G, s);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime.
EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace

cudaError_t encode_cache_maps(const CacheView& c, int Hkv, int D, CUtensorMap* k, CUtensorMap* v) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn) return cudaErrorNotSupported;
  const uint64_t rows = static_cast<uint64_t>(c.n_rows) * Hkv * (c.paged ? c.P : c.R);
  if (rows == 0 || rows > 0x7fffffffull) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  const cuuint32_t box[2] = {64, kGroup};
  const cuuint32_t estride[2] = {1, 1};
  for (int i = 0; i < 2; ++i) {
    const CUresult r = fn(i ? v : k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, i ? c.v : c.k, dims, strides,
                          box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

cudaError_t launch_decode_split(const SplitArgs& a, int D, int G, cudaStream_t s) {
  const int GP = decode_group_pad(G);
  if (a.B * a.Hkv > kMaxUnits) return cudaErrorNotSupported;
  if (D == 256) {
    if (GP == 4) return split_dispatch_paged<256, 1>(a, G, s);
    if (GP == 8) return split_dispatch_paged<256, 2>(a, G, s);
  } else if (D == 128) {
    if (GP == 4) return split_dispatch_paged<128, 1>(a, G, s);
    if (GP == 8) return split_dispatch_paged<128, 2>(a, G, s);
  }
  return cudaErrorNotSupported;
}

int decode_split_tile_keys(int D, int G) {
  if (decode_group_pad(G) == 0 || (D != 128 && D != 256)) return 0;
  return 256 / D * kGroup;
}

int decode_split_ctas_per_sm(int D, int G) {
  const int GP = decode_group_pad(G);
  int smem = 0;
  if (D == 256) smem = GP == 4 ? Geo<256, 1>::SMEM_MAX : GP == 8 ? Geo<256, 2>::SMEM_MAX : 0;
  if (D == 128) smem = GP == 4 ? Geo<128, 1>::SMEM_MAX : GP == 8 ? Geo<128, 2>::SMEM_MAX : 0;
  if (smem == 0) return 0;
  // 228 KB of shared memory per SM; 1 KB reserved and the static block-scan scratch per CTA
  const int per_sm = 233472 / (smem + 1024 + 64);
  return per_sm > 2 ? 2 : per_sm;
}

int decode_max_units() { return kMaxUnits; }

cudaError_t launch_decode_combine(const CombineArgs& a, int D, int G, cudaStream_t s) {
  const int GP = decode_group_pad(G);
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
