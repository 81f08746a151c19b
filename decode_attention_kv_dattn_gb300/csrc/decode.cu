// Decode attention in one launch per call: RoPE of the new token, the pass
// over the cached keys, the join of the new token in score space, the output
// gate, the fp32 store and the write-back of the new K/V entry.
//
// Method ("vllm-omni commits", score-space join commit): the cached keys (n of
// them) and the new key are scored separately and their score vectors meet in
// one softmax; nothing cache-sized is copied, and the new K/V entry is written
// into its slot afterwards. A ring's slots need no reordering (softmax is
// order-free, cached keys carry their own rotary phase); unwritten slots are
// masked. Per-layer-type RoPE and the head-wise sigmoid gate follow the Spark
// model commit of the same page; grouped-query attention shares each KV head's
// loads among its G query heads (talker export commit). Splitting the keys
// over many CTAs and merging their partial softmax states follows "TensorFold
// PR #608" (the grid must fill the GPU; a merge must not be a chain of
// dependent loads).
//
// GB300 design.
//  * Work split (stream-K). A "unit" is one (stream, KV head). Its cached keys
//    are visited in groups of 16 rows: 16-row runs of a page (a page of P
//    rows gives ceil(P / 16) groups), or every 16-slot block of the ring's
//    physical slots, in slot order (the unwritten slots masked: a ring
//    layer's split then needs none of its metadata, and its first copies go
//    out before that metadata has arrived). A stage tile is 256 / D groups
//    (16 KB of K and V). All units'
//    tiles are laid end to end and the grid - one CTA per SM - cuts that
//    sequence into equal contiguous ranges, so every CTA moves the same number
//    of bytes whatever the mix of lengths. Each piece of a unit inside one CTA
//    (a "segment") leaves one partial softmax state (m, l, o) in global
//    memory; the CTA that finishes a unit's last segment (a per-unit counter)
//    merges them with the new token's score, applies the gate, stores the
//    output and writes the new entry back - after every read of the cache.
//  * RoPE. A helper warp rotates each unit's G query heads one segment ahead
//    (fp32, pre-scaled by log2(e)/sqrt(D)); the cos/sin of each pair come from
//    an exact fixed-point phase and an fp32 polynomial (rope_cos_sin). It
//    rotates the new key with the same cos/sin and rounds it to the bf16
//    nearest the exact rotation (fp32 error terms, an integer fallback near a
//    bf16 midpoint: bf16_dot2) - the entry that is scored and stored.
//  * Loads. Each warp owns a ring of NS stage buffers. One lane issues tensor
//    TMA copies (16 rows of a group, 128-byte swizzle: one 3D box for both
//    64-dim regions at D = 128, one 2D box per region at D = 256) for the
//    warp's tile NS ahead, with
//    completion counted in bytes on the stage's mbarrier; the ring keeps
//    streaming across segment boundaries. The rows of each group and its
//    valid-row mask (past a unit's length, past a page, outside a ring's valid
//    slots, or zero-filled past the pool) are worked out by the whole warp for
//    32 tiles at a time, a window ahead, so that no page-table load sits on the
//    issue path. Invalid rows get -inf scores and zeroed V rows.
//  * Math on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate).
//    The KV stream is HBM-bound at G flops per byte; the tensor cores are used
//    because they cut the instructions per byte about tenfold against fp32
//    FMAs, which otherwise limit the issue rate. Per group of 16 keys:
//      S^T (16 keys x 8 cols) = K (16 x D) . Q^T (D x 8 cols)
//      O^T (D x 8 cols)      += V^T (D x 16) . P^T (16 x 8 cols)
//    The 8 (or 2 x 8) columns hold each query head twice: once as the bf16
//    rounding of the rotated q, once as the bf16 rounding of what is left
//    ("hi" and "lo"), so q keeps 16 significant bits; the two score columns of
//    a head are added. The probabilities are split into hi and lo bf16 parts
//    the same way, and the two output columns of a head are added at the end.
//    K and V enter the tensor cores exactly (they are bf16). The score
//    fragment becomes the PV operand in registers (movmatrix transposes);
//    online softmax in base 2 runs on the score fragment, and the output is
//    rescaled only when some head's running maximum moved.
#include "bf16_exact.h"
#include "common.cuh"
#include "qk_norm.cuh"
#include "round_f64.h"
#include "mma.cuh"

namespace dattn {

namespace {

constexpr unsigned kFull = 0xffffffffu;
// Streaming warps of a kernel variant: 4 with 16 KB stage tiles, or 7 with
// 8 KB tiles for E4M3 at D = 256, so that every SM sub-partition runs two
// warps (7 streaming + the helper; 255 registers a thread still fit each
// sub-partition's register file) that hide one another's conversion chains:
// 128k x 8 streams 241 -> 230 us per call. At D = 128 the same split measured
// slower (bf16 paged batch 106 -> 121 us, E4M3 133 -> 149 us).
template <int D, int NT, bool F8>
constexpr int stream_warps() {
  return (F8 && D == 256) ? 7 : 4;
}
// Stage tiles per streaming warp, and bytes of K and V in one stage tile.
template <int D, int NT, bool F8>
constexpr int stage_count() {
  return 3;
}
template <int D, int NT, bool F8>
constexpr int stage_bytes() {
  return stream_warps<D, NT, F8>() > 4 ? 8192 : 16384;
}
constexpr int kMaxUnits = 512;           // (stream, KV head) units per call
constexpr int kGroup = 16;               // keys per MMA group
constexpr int kBoxBytes = kGroup * 128;  // one TMA box: 16 rows x 64 bf16
constexpr int kWin = 32;                 // tiles per prefetch window (one per lane)
constexpr int64_t kPrefetchLines = 1 << 15;  // largest page table (128-byte lines) put in L2 at start
// Fixed cost of one segment of a unit in the stream-K split, in stage tiles of
// one CTA: a segment boundary takes about as long as streaming this many
// tiles with all warps.
#ifndef DATTN_SEGMENT_COST
#define DATTN_SEGMENT_COST 12
#endif
constexpr int kSegmentCost = DATTN_SEGMENT_COST;
#ifndef DATTN_MERGE_BATCH
#define DATTN_MERGE_BATCH 8
#endif
constexpr int kMergeBatch = DATTN_MERGE_BATCH;  // partials read per round trip by a unit's final merge
// Largest excess (percent) of the biggest piece over a fair share of the tiles
// for which the split cuts every unit into equal pieces instead of stream-K.
#ifndef DATTN_PIECES_SLACK
#define DATTN_PIECES_SLACK 25
#endif
constexpr int kPiecesSlack = DATTN_PIECES_SLACK;
// TMA boxes per 16-row group: at D = 128 one 3D box takes both 64-dim regions
// (measured faster); at D = 256 one 2D box per region (the single 8 KB box
// measured slower on the 16-token-page and ring layers of the hybrid step).
template <int D>
constexpr bool kGroupBox = D == 128;

template <int D, int NT, bool F8 = false>
struct Geo {
  static constexpr int W = stream_warps<D, NT, F8>();  // streaming warps; the helper is warp W
  static constexpr int THREADS = (W + 1) * 32;
  static constexpr int GP = 4 * NT;                  // heads per partial slot
  static constexpr int KSTEPS = D / 16;              // MMA k-steps of a score, m-tiles of an output
  static constexpr int ROWB = F8 ? D : 2 * D;        // bytes of one cached row (bf16, or E4M3)
  static constexpr int BOXES = ROWB / 128;           // 128-byte boxes per 16-row group of K (or V)
  static constexpr int GBYTES = BOXES * kBoxBytes;   // K (or V) bytes of one group
  static constexpr int KG = stage_bytes<D, NT, F8>() / (2 * 16 * ROWB);  // groups per stage tile
  static constexpr int KHALF = KG * GBYTES;          // K part of a stage; V follows
  static constexpr int STAGE = 2 * KHALF;
  static constexpr int NS = stage_count<D, NT, F8>();
  // mbarriers: [W][NS] stages, 2 input slots, then the four hand-offs
  // between the streaming warps and the helper
  static constexpr int NBAR = W * NS + 2 + 4;
  // offsets from the 1024-byte aligned base of dynamic shared memory
  static constexpr int BAR_OFF = W * NS * STAGE;
  static constexpr int INBAR_OFF = BAR_OFF + W * NS * 8;
  static constexpr int PREP_FULL_OFF = INBAR_OFF + 16;   // q of the next segment is in qs
  static constexpr int PREP_EMPTY_OFF = INBAR_OFF + 24;  // every streaming warp has read qs
  static constexpr int MERGE_FULL_OFF = INBAR_OFF + 32;  // every warp's state is in its buffer
  static constexpr int MERGE_EMPTY_OFF = INBAR_OFF + 40; // the helper has read the states
  static constexpr int ML_OFF = BAR_OFF + NBAR * 8;               // float [W][2*GP]
  static constexpr int SLOT_OFF = ML_OFF + W * 2 * GP * 4;   // int [W]
  static constexpr int FLAG_OFF = SLOT_OFF + W * 4;          // int: "this CTA combines"
  static constexpr int CS_OFF = (FLAG_OFF + 4 + 15) / 16 * 16;    // float2 [D/2]: cos, sin
  static constexpr int QS_OFF = CS_OFF + D / 2 * 8;               // float [GP][D]: rotated q
  static constexpr int WROW_OFF = QS_OFF + GP * D * 4;            // int [W][2][kWin*KG]
  static constexpr int WMASK_OFF = WROW_OFF + W * 2 * kWin * KG * 4;
  static constexpr int STEP_OFF = WMASK_OFF + W * 2 * kWin * KG * 4;  // uint64 [D/2]: RoPE steps
  // input slot: q [GP][D] bf16, k_new [D], v_new [D] (one bulk copy each),
  // then the new token worked out from them: K entry [D] bf16, scores [GP],
  // sigmoid(gate) [GP]
  static constexpr int IN_Q = 0;
  static constexpr int IN_K = GP * D * 2;
  static constexpr int IN_V = IN_K + D * 2;
  static constexpr int IN_KH = IN_V + D * 2;
  static constexpr int IN_SN = IN_KH + D * 2;
  static constexpr int IN_SIG = IN_SN + GP * 4;
  static constexpr int IN_WB = (IN_SIG + GP * 4 + 7) / 8 * 8;  // int64: the new entry's pool offset
  static constexpr int IN_BYTES = (IN_WB + 8 + 15) / 16 * 16;
  static constexpr int IN_OFF = (STEP_OFF + D / 2 * 8 + 15) / 16 * 16;  // 2 input slots
  static constexpr int TAB_OFF = IN_OFF + 2 * IN_BYTES;
  static constexpr int SMEM_MAX = 1024 + TAB_OFF + (4 * kMaxUnits + 1) * 4;  // P, N, ring head/row
  static_assert(D == 128 || D == 256, "head_dim");
  static_assert(KG >= 1 && KG * 2 * 16 * ROWB == STAGE, "a stage tile holds whole 16-row groups");
  static_assert(GP * D * 4 <= STAGE, "a stage buffer holds one warp's partial output");
  static_assert(NS < kWin, "issue runs at most one window ahead");
  static_assert(SMEM_MAX <= 232448, "shared memory per CTA");
};

// Cached keys of call row b (the same for all its KV heads). Bad metadata is
// reported (once per row) and yields no keys.
template <bool PAGED>
__device__ __forceinline__ int unit_length(const CacheView& c, int b, int max_len, bool report,
                                           int* err) {
  static_assert(PAGED, "ring units: ring_length");
  int n = c.seq_len[b];
  const int cap = min(max_len, c.bt_stride * c.P);
  if (n < 0 || n > cap) {
    if (report) raise_error(err, ERR_LENGTH);
    n = n < 0 ? 0 : cap;
  }
  return n;
}

// Valid slots of a ring from its metadata (cache row, head slot, count): 0,
// and an index error, when any of them is out of range.
__device__ __forceinline__ int ring_length(const CacheView& c, int row, int head, int cnt, bool report, int* err) {
  if (row < 0 || row >= c.n_rows || head < 0 || head >= c.R || cnt < 0 || cnt > c.R) {
    if (report) raise_error(err, ERR_INDEX);
    return 0;
  }
  return cnt;
}

// First slot of a ring holding `n` valid slots before `head`.
__device__ __forceinline__ int ring_start(int head, int n, int R) {
  return head - n < 0 ? head - n + R : head - n;
}

// 16-row groups of a paged unit with n cached keys.
__device__ __forceinline__ int paged_groups(const CacheView& c, int n) {
  if (n <= 0) return 0;
  const int gpp = (c.P + kGroup - 1) / kGroup;
  const int full = n / c.P, rest = n - full * c.P;
  return full * gpp + (rest + kGroup - 1) / kGroup;
}

// Bits r of the valid rows [lo, hi) of a 16-row group (empty when hi <= lo).
__device__ __forceinline__ uint32_t row_bits(int lo, int hi) {
  lo = max(lo, 0);
  hi = min(hi, kGroup);
  if (hi <= lo) return 0u;
  return ((1u << (hi - lo)) - 1u) << lo;
}

// Work on one unit's inputs and outputs is done by a team: the helper warp
// (NTH = 32, t = lane) for segment ends in the middle of a CTA's range, or the
// whole CTA (NTH = kThreads, t = threadIdx.x) for its last one.
template <int NTH>
__device__ __forceinline__ void team_sync() {
  if constexpr (NTH == 32) __syncwarp(); else __syncthreads();
}

// QK-norm of a unit's staged rows in place, before they are rotated: its G
// query rows (weights a.q_norm) and its new key (a.k_norm), one warp per row.
// Ends with a team barrier.
template <int D, int NTH>
__device__ __forceinline__ void norm_staged(const DecodeArgs& a, uint16_t* q, uint16_t* k, int t) {
  constexpr int W = NTH / 32;
  const int w = t >> 5, lane = t & 31;
  for (int row = w; row <= a.G; row += W) {
    const uint16_t* wt = row < a.G ? a.q_norm : a.k_norm;
    if (!wt) continue;
    uint16_t* x = row < a.G ? q + row * D : k;
    const double inv = qk_norm_inv(x, D, a.norm_eps, lane);
    for (int d = lane; d < D; d += 32) x[d] = qk_norm_apply(x[d], wt[d], inv);
  }
  fence_proxy_async_smem();  // the slot is refilled by bulk copies later
  team_sync<NTH>();
}

// Rotate the G query heads of a unit (src: its staged q rows [G][D]) at
// position pos into qs[GP][D] (fp32, pre-scaled; heads >= G are zero) and keep
// each pair's cos/sin in cs.
template <int D, int GP, int NTH>
__device__ __forceinline__ void prep_q(const DecodeArgs& a, const uint16_t* src, int pos, const uint64_t* step,
                                       float* qs, float2* cs, int t) {
  const int G = a.G, half = a.r / 2;
  for (int p = t; p < D / 2; p += NTH) {
    const int d0 = p < half ? p : a.r + 2 * (p - half);
    const int d1 = p < half ? p + half : d0 + 1;
    float c = 1.f, s = 0.f;
    if (p < half) rope_cos_sin(pos, step[p], c, s);
    cs[p] = make_float2(c, s);
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

// The new token of a unit from its input slot: its K entry (the bf16 nearest
// to the exact rotation with the cos/sin in cs - the value that is scored and
// stored), its score per head (base 2, with the rotated q in qs) and the
// heads' sigmoid(gate) (gate_raw: the bf16 logit of head t, for t < G), all
// into the slot. Starts after cs and qs are complete for the team; ends with a
// team barrier.
template <int D, int GP, int NTH>
__device__ __forceinline__ void prep_token(const DecodeArgs& a, const float* qs, const float2* cs, uint8_t* slot,
                                           uint16_t gate_raw, int t) {
  using Gm = Geo<D, GP / 4>;
  const int G = a.G, half = a.r / 2;
  const uint16_t* ksrc = reinterpret_cast<const uint16_t*>(slot + Gm::IN_K);
  uint16_t* kh = reinterpret_cast<uint16_t*>(slot + Gm::IN_KH);
  float* sn = reinterpret_cast<float*>(slot + Gm::IN_SN);
  float* sig = reinterpret_cast<float*>(slot + Gm::IN_SIG);
  if (t < G) sig[t] = a.gate ? 1.f / (1.f + expf(-bf16_to_f32(gate_raw))) : 1.f;
  // E4M3 cache: the entry and v_new are stored (and scored) as the E4M3 bytes
  // nearest entry / k_scale and v_new / v_scale, at IN_KH (K, then V)
  uint8_t* k8 = slot + Gm::IN_KH;
  const uint16_t* vsrc = reinterpret_cast<const uint16_t*>(slot + Gm::IN_V);
  for (int e = t; e < D; e += NTH) {
    uint16_t v = ksrc[e];
    if (e < half) {
      const float2 q = cs[e];  // x c - y s with x = k[e], y = k[e + half]
      v = bf16_dot2(ksrc[e], __float_as_uint(q.x), ksrc[e + half], __float_as_uint(q.y) ^ 0x80000000u);
    } else if (e < a.r) {
      const float2 q = cs[e - half];  // y c + x s with y = k[e], x = k[e - half]
      v = bf16_dot2(ksrc[e], __float_as_uint(q.x), ksrc[e - half], __float_as_uint(q.y));
    }
    if (a.f8) {
      k8[e] = e4m3_from_f64(static_cast<double>(bf16_to_f32(v)) / static_cast<double>(a.k_scale));
      k8[D + e] = e4m3_from_f64(static_cast<double>(bf16_to_f32(vsrc[e])) / static_cast<double>(a.v_scale));
    } else {
      kh[e] = v;
    }
  }
  team_sync<NTH>();
  constexpr int W = NTH / 32;
  const int w = t >> 5, lane = t & 31;
  for (int g = w; g < G; g += W) {
    float dot = 0.f;
    for (int d = lane; d < D; d += 32)
      dot = fmaf(qs[g * D + d], a.f8 ? e4m3_to_f32(k8[d]) : bf16_to_f32(kh[d]), dot);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) dot += __shfl_xor_sync(kFull, dot, o);
    if (lane == 0) sn[g] = dot;
  }
  team_sync<NTH>();
}

// Running merge of softmax states (max m, sum l, output slice o) over the
// dims of one head: starts from the new token (m = its score, l = 1, o = v).
struct Merge8 {
  float M, L, o[8];
  __device__ __forceinline__ void add(float m, float l, const float (&x)[8]) {
    const float Mn = fmaxf(M, m);
    const float al = exp2_fast(M - Mn), be = exp2_fast(m - Mn);
    L = fmaf(L, al, l * be);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = fmaf(o[i], al, x[i] * be);
    M = Mn;
  }
};

// Where unit (b, j)'s new entry goes: its element offset in the K and V
// pools (bytes for E4M3), or -1 when the metadata is out of range (a bad
// page is reported here; a bad ring was reported when the unit table was read).
template <bool PAGED>
__device__ __forceinline__ int64_t write_back_offset(const DecodeArgs& a, int b, int j, int D) {
  const CacheView& c = a.c;
  if constexpr (PAGED) {
    const int n = min(max(c.seq_len[b], 0), min(a.max_len, c.bt_stride * c.P));
    const int pi = n / c.P;
    const int pg = pi < c.bt_stride ? c.block_table[static_cast<int64_t>(b) * c.bt_stride + pi] : -1;
    if (pg >= 0 && pg < c.n_rows) return ((static_cast<int64_t>(pg) * a.Hkv + j) * c.P + n % c.P) * D;
    raise_error(a.err, ERR_INDEX);
    return -1;
  } else {
    const int row = c.stream_rows ? c.stream_rows[b] : b;
    const int head = c.ring_head[b], cnt = c.ring_count[b];
    if (row < 0 || row >= c.n_rows || head < 0 || head >= c.R || cnt < 0 || cnt > c.R) return -1;
    return ((static_cast<int64_t>(row) * a.Hkv + j) * c.R + head) * D;
  }
}

// Output and write-back of unit u = (b, j) once all of its segments are done.
// Each thread takes 8 consecutive dims of one head; `states(g, d, mg)` folds
// the unit's segment states for head g, dims d..d+7 into mg. Needs the new
// token in the unit's input slot. No barrier at the end.
template <int D, int GP, bool PAGED, int NTH, typename States>
__device__ __forceinline__ void finish_unit(const DecodeArgs& a, int u, const uint8_t* slot, int t,
                                            States states) {
  using Gm = Geo<D, GP / 4>;
  const int Hkv = a.Hkv, G = a.G, Hq = Hkv * G;
  const int b = u / Hkv, j = u - b * Hkv;
  const CacheView& c = a.c;
  const uint16_t* vsrc = reinterpret_cast<const uint16_t*>(slot + Gm::IN_V);
  const uint16_t* kh = reinterpret_cast<const uint16_t*>(slot + Gm::IN_KH);
  const float* sn = reinterpret_cast<const float*>(slot + Gm::IN_SN);
  const float* sig = reinterpret_cast<const float*>(slot + Gm::IN_SIG);
  for (int e = t * 8; e < G * D; e += NTH * 8) {
    const int g = e / D, d = e - g * D;
    Merge8 mg;
    mg.M = sn[g];
    mg.L = 1.f;
    if (a.f8) {
      const uint8_t* v8 = slot + Gm::IN_KH + D;  // the new token's V as stored
#pragma unroll
      for (int i = 0; i < 8; ++i) mg.o[i] = e4m3_to_f32(v8[d + i]) * a.v_scale;
    } else {
      const uint4 vw = *reinterpret_cast<const uint4*>(vsrc + d);
      mg.o[0] = bf16_lo(vw.x); mg.o[1] = bf16_hi(vw.x);
      mg.o[2] = bf16_lo(vw.y); mg.o[3] = bf16_hi(vw.y);
      mg.o[4] = bf16_lo(vw.z); mg.o[5] = bf16_hi(vw.z);
      mg.o[6] = bf16_lo(vw.w); mg.o[7] = bf16_hi(vw.w);
    }
    states(g, d, mg);
    const float scale = sig[g] / mg.L;
    float* dst = a.out + (static_cast<int64_t>(b) * Hq + j * G + g) * D + d;
    *reinterpret_cast<float4*>(dst) = make_float4(mg.o[0] * scale, mg.o[1] * scale, mg.o[2] * scale, mg.o[3] * scale);
    *reinterpret_cast<float4*>(dst + 4) = make_float4(mg.o[4] * scale, mg.o[5] * scale, mg.o[6] * scale, mg.o[7] * scale);
  }
  // write-back of the new entry: every segment of this unit has finished
  // reading; its target was worked out when the unit's inputs were prepared
  if (a.write_back) {
    const int64_t wb = *reinterpret_cast<const int64_t*>(slot + Gm::IN_WB);
    if (wb >= 0 && a.f8) {
      // E4M3 rows: wb counts elements, which are bytes here
      const uint8_t* k8 = slot + Gm::IN_KH;
      for (int d = t * 16; d < D; d += NTH * 16) {
        *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(c.k) + wb + d) = *reinterpret_cast<const uint4*>(k8 + d);
        *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(c.v) + wb + d) =
            *reinterpret_cast<const uint4*>(k8 + D + d);
      }
    } else if (wb >= 0) {
      for (int d = t * 8; d < D; d += NTH * 8) {
        *reinterpret_cast<uint4*>(c.k + wb + d) = *reinterpret_cast<const uint4*>(kh + d);
        *reinterpret_cast<uint4*>(c.v + wb + d) = *reinterpret_cast<const uint4*>(vsrc + d);
      }
    }
  }
}

// The streaming warps' states of one segment (merge buffers: warp w's stage
// SLOT[w], or none when SLOT[w] < 0) folded into mg for head g, dims d..d+7.
template <int D, int NT, bool F8>
__device__ __forceinline__ void fold_warps(const uint8_t* smem, const float* ML, const int* SLOT, int g, int d,
                                           Merge8& mg) {
  using Gm = Geo<D, NT, F8>;
  constexpr int kWarps = Gm::W;
  constexpr int GP = Gm::GP;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int st = SLOT[w];
    if (st < 0) continue;
    const float* os = reinterpret_cast<const float*>(smem + (w * Gm::NS + st) * Gm::STAGE) + g * D + d;
    const float4 x0 = *reinterpret_cast<const float4*>(os);
    const float4 x1 = *reinterpret_cast<const float4*>(os + 4);
    const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    mg.add(ML[w * 2 * GP + g], ML[w * 2 * GP + GP + g], x);
  }
}

// The streaming warps' states of one segment merged into the partial slot
// dst: o[GP][D] (relative to the merged maximum), then m[GP], l[GP]. No
// barrier at the end.
template <int D, int NT, bool F8, int NTH>
__device__ __forceinline__ void write_partial(const uint8_t* smem, const float* ML, const int* SLOT, float* dst,
                                              int t) {
  using Gm = Geo<D, NT, F8>;
  constexpr int kWarps = Gm::W;
  constexpr int GP = Gm::GP;
  for (int e = t * 8; e < GP * D; e += NTH * 8) {
    const int h = e / D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      if (SLOT[w] >= 0) M = fmaxf(M, ML[w * 2 * GP + h]);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const int st = SLOT[w];
        if (st < 0) continue;
        const float f = exp2_fast(ML[w * 2 * GP + h] - M);
        const float* os = reinterpret_cast<const float*>(smem + (w * Gm::NS + st) * Gm::STAGE) + e;
        const float4 x0 = *reinterpret_cast<const float4*>(os);
        const float4 x1 = *reinterpret_cast<const float4*>(os + 4);
        acc[0] = fmaf(f, x0.x, acc[0]); acc[1] = fmaf(f, x0.y, acc[1]);
        acc[2] = fmaf(f, x0.z, acc[2]); acc[3] = fmaf(f, x0.w, acc[3]);
        acc[4] = fmaf(f, x1.x, acc[4]); acc[5] = fmaf(f, x1.y, acc[5]);
        acc[6] = fmaf(f, x1.z, acc[6]); acc[7] = fmaf(f, x1.w, acc[7]);
      }
    }
    *reinterpret_cast<float4*>(dst + e) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(dst + e + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  for (int h = t; h < GP; h += NTH) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      if (SLOT[w] >= 0) M = fmaxf(M, ML[w * 2 * GP + h]);
    float L = 0.f;
    if (M != -INFINITY)
#pragma unroll
      for (int w = 0; w < kWarps; ++w)
        if (SLOT[w] >= 0) L = fmaf(exp2_fast(ML[w * 2 * GP + h] - M), ML[w * 2 * GP + GP + h], L);
    dst[GP * D + h] = M;
    dst[GP * D + GP + h] = L;
  }
}

// Bulk copies (issued by the calling thread) of unit u's q, k_new and v_new
// rows into input slot n & 1, counted on that slot's mbarrier; the first
// staging of a CTA (n == 0) also brings the layer's RoPE phase steps (the
// table is allocated in whole 16-byte units).
template <int D, int GP>
__device__ __forceinline__ void issue_stage(const DecodeArgs& a, int u, int n, uint32_t inbar, uint8_t* in_slots,
                                            uint64_t* step) {
  using Gm = Geo<D, GP / 4>;
  const int Hkv = a.Hkv, G = a.G;
  const int b = u / Hkv, j = u - b * Hkv;
  const uint32_t bar = inbar + 8 * (n & 1);
  const uint32_t dst = smem_addr(in_slots + (n & 1) * Gm::IN_BYTES);
  const uint32_t qbytes = static_cast<uint32_t>(G) * D * 2;
  const uint32_t sbytes = n == 0 ? (static_cast<uint32_t>(a.r / 2) * 8u + 15u) / 16u * 16u : 0u;
  const uint64_t pol = l2_evict_first_policy();
  mbar_arrive_expect_tx(bar, qbytes + 4u * D + sbytes);
  if (sbytes) bulk_copy_g2s(smem_addr(step), a.rope_step, sbytes, bar, pol);
  bulk_copy_g2s(dst + Gm::IN_Q, a.q + (static_cast<int64_t>(b) * Hkv + j) * G * D, qbytes, bar, pol);
  bulk_copy_g2s(dst + Gm::IN_K, a.k_new + (static_cast<int64_t>(b) * Hkv + j) * D, 2u * D, bar, pol);
  bulk_copy_g2s(dst + Gm::IN_V, a.v_new + (static_cast<int64_t>(b) * Hkv + j) * D, 2u * D, bar, pol);
}

// Folds the partial slots base[k * slot_stride] (k in [k0, k1), where ok(k))
// into mg, kMergeBatch slots' loads in flight at a time, for head g, dims
// d..d+7. Slots with no valid key (m = -inf) are skipped.
template <int D, int GP, typename Ok, typename Slot>
__device__ __forceinline__ void fold_slots(const float* part, int k0, int k1, Ok ok, Slot slot_of, int g, int d,
                                           Merge8& mg) {
  constexpr int stride = GP * (D + 2);
  for (int kb = k0; kb < k1; kb += kMergeBatch) {
    float m[kMergeBatch], l[kMergeBatch], x[kMergeBatch][8];
#pragma unroll
    for (int q = 0; q < kMergeBatch; ++q) {
      const int k = kb + q;
      m[q] = -INFINITY;
      l[q] = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) x[q][i] = 0.f;
      if (k < k1 && ok(k)) {
        const float* pk = part + static_cast<int64_t>(slot_of(k)) * stride;
        m[q] = __ldcg(pk + GP * D + g);
        l[q] = __ldcg(pk + GP * D + GP + g);
        const float4 y0 = __ldcg(reinterpret_cast<const float4*>(pk + g * D + d));
        const float4 y1 = __ldcg(reinterpret_cast<const float4*>(pk + g * D + d + 4));
        x[q][0] = y0.x; x[q][1] = y0.y; x[q][2] = y0.z; x[q][3] = y0.w;
        x[q][4] = y1.x; x[q][5] = y1.y; x[q][6] = y1.z; x[q][7] = y1.w;
      }
    }
#pragma unroll
    for (int q = 0; q < kMergeBatch; ++q)
      if (m[q] != -INFINITY) mg.add(m[q], l[q], x[q]);
  }
}

// A unit cut into many pieces (one per CTA: a long stream on a GPU of many
// SMs; 76 pieces at 1 x 131,072) is merged in two levels, so that its final
// merge is not one CTA reading every partial (~17 us for 76 of them): the CTA
// that finishes the last piece of a group of kMergeBatch pieces merges the
// group into the slot of its first piece (per-group counters follow the unit
// counters), and the CTA that finishes the last group merges the groups'
// results with the new token. Called by the whole CTA after its piece's
// partial is stored and published.
template <int D, int GP, bool PAGED, int NTH, typename WaitPrev>
__device__ void merge_in_groups(const DecodeArgs& a, int U, int pieces, int u, int cta, int unit_tiles,
                                const uint8_t* slot, int* flag, int t, WaitPrev wait_prev) {
  constexpr int stride = GP * (D + 2);
  constexpr int IPT = (GP * D / 8 + NTH - 1) / NTH;  // 8-dim items per thread
  const int S = pieces;
  auto piece_ok = [&](int k) { return k < S && (k + 1) * unit_tiles / pieces > k * unit_tiles / pieces; };
  auto piece_slot = [&](int k) { return u * pieces + k; };
  auto group_first = [&](int kb) {  // first piece of group [kb, kb + kMergeBatch) with tiles, or -1
    for (int k = kb; k < min(S, kb + kMergeBatch); ++k)
      if (piece_ok(k)) return k;
    return -1;
  };
  const int kb = (cta - u * pieces) / kMergeBatch * kMergeBatch, ke = min(S, kb + kMergeBatch);
  int n_in = 0;
  for (int k = kb; k < ke; ++k) n_in += piece_ok(k);
  int* gcount = a.counters + U + piece_slot(kb);
  if (t == 0) *flag = atomicAdd(gcount, 1) == n_in - 1;
  __syncthreads();
  if (!*flag) return;
  __threadfence();
  // ---- the group, into the slot of its first piece: o first (each thread
  // reads and writes only its own items' dims), m and l once every thread
  // has read the group's
  float* gdst = a.part + static_cast<int64_t>(piece_slot(group_first(kb))) * stride;
  float gM[IPT], gL[IPT];
#pragma unroll
  for (int i = 0; i < IPT; ++i) {
    gM[i] = -INFINITY;
    gL[i] = 0.f;
    const int e = t * 8 + i * NTH * 8;
    if (e < a.G * D) {
      const int g = e / D, d = e - g * D;
      Merge8 r;
      r.M = -INFINITY;
      r.L = 0.f;
#pragma unroll
      for (int x = 0; x < 8; ++x) r.o[x] = 0.f;
      fold_slots<D, GP>(a.part, kb, ke, piece_ok, piece_slot, g, d, r);
      gM[i] = r.M;
      gL[i] = r.L;
      *reinterpret_cast<float4*>(gdst + g * D + d) = make_float4(r.o[0], r.o[1], r.o[2], r.o[3]);
      *reinterpret_cast<float4*>(gdst + g * D + d + 4) = make_float4(r.o[4], r.o[5], r.o[6], r.o[7]);
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < IPT; ++i) {
    const int e = t * 8 + i * NTH * 8;
    if (e < a.G * D && e % D == 0) {
      gdst[GP * D + e / D] = gM[i];
      gdst[GP * D + GP + e / D] = gL[i];
    }
  }
  if (t == 0) *gcount = 0;
  __threadfence();
  __syncthreads();
  // ---- count this group; the CTA finishing the unit's last group combines
  int n_groups = 0;
  for (int k = 0; k < S; k += kMergeBatch) n_groups += group_first(k) >= 0;
  if (t == 0) *flag = atomicAdd(a.counters + u, 1) == n_groups - 1;
  __syncthreads();
  if (!*flag) return;
  __threadfence();
  wait_prev();
  auto group_ok = [&](int gi) { return group_first(gi * kMergeBatch) >= 0; };
  auto group_slot = [&](int gi) { return piece_slot(group_first(gi * kMergeBatch)); };
  const int ng = (S + kMergeBatch - 1) / kMergeBatch;
  finish_unit<D, GP, PAGED, NTH>(a, u, slot, t, [&](int g, int d, Merge8& mg) {
    fold_slots<D, GP>(a.part, 0, ng, group_ok, group_slot, g, d, mg);
  });
  if (t == 0) a.counters[u] = 0;
  __syncthreads();
}

// End of one segment of unit u, whose streaming warps' states are in their
// merge buffers. When the unit lies wholly in this CTA, its output and
// write-back follow from those states; otherwise they are merged into the
// segment's partial slot, and the CTA finishing the unit's last segment (a
// per-unit counter) merges all of its partials. `release()` runs once the
// merge buffers have been read; `wait_prev()` before the first output store.
template <int D, int NT, bool PAGED, bool F8, int NTH, typename WaitPrev, typename Release>
__device__ void end_segment(const DecodeArgs& a, const Split& sp, int pieces, int u, bool first_seg, int cta,
                            const uint8_t* smem, const float* ML, const int* SLOT, const uint8_t* slot, int* flag,
                            int t, WaitPrev wait_prev, Release release) {
  using Gm = Geo<D, NT>;
  constexpr int GP = Gm::GP;
  const int NC = sp.NC, p0 = sp.P[u], p1 = sp.P[u + 1];
  int c_lo = 0, c_hi = 0, first_slot = 0, nseg, S;
  if (pieces) {
    nseg = min(pieces, p1 - p0);
    S = pieces;
  } else {
    nseg = unit_segments(sp, p0, p1, u, c_lo, c_hi, first_slot);
    S = c_hi - c_lo + 1;
  }
  if (nseg == 1) {
    // the whole unit lies in this CTA: the warps' states go straight into the output
    wait_prev();
    finish_unit<D, GP, PAGED, NTH>(a, u, slot, t, [&](int g, int d, Merge8& mg) {
      fold_warps<D, NT, F8>(smem, ML, SLOT, g, d, mg);
    });
    team_sync<NTH>();
    release();
    return;
  }
  const int pslot = first_seg ? cta : NC + u;
  write_partial<D, NT, F8, NTH>(smem, ML, SLOT, a.part + static_cast<int64_t>(pslot) * (GP * (D + 2)), t);
  __threadfence();
  team_sync<NTH>();
  release();
  if constexpr (NTH != 32) {
    if (pieces && S > 2 * kMergeBatch) {
      merge_in_groups<D, GP, PAGED, NTH>(a, sp.U, pieces, u, cta, p1 - p0, slot, flag, t, wait_prev);
      return;
    }
  }
  // count this segment; the team finishing the unit's last segment combines it
  int last;
  if constexpr (NTH == 32) {
    last = t == 0 ? atomicAdd(a.counters + u, 1) == nseg - 1 : 0;
    last = __shfl_sync(kFull, last, 0);
  } else {
    if (t == 0) *flag = atomicAdd(a.counters + u, 1) == nseg - 1;
    __syncthreads();
    last = *flag;
  }
  if (!last) return;
  __threadfence();
  wait_prev();
  // candidate k: the partial slot of the k-th CTA of the unit's span, and
  // whether it holds tiles of the unit
  auto cand_slot = [&](int k) { return pieces ? u * pieces + k : (k == 0 ? first_slot : c_lo + k); };
  auto cand_ok = [&](int k) -> bool {
    if (k >= S) return false;
    if (pieces) return (k + 1) * (p1 - p0) / pieces > k * (p1 - p0) / pieces;
    // candidate k > 0 is the first segment of CTA c_lo + k, unless that CTA got no tiles
    return k == 0 || sp.has_tiles_inside(c_lo + k);
  };
  const int stride = GP * (D + 2);
  finish_unit<D, GP, PAGED, NTH>(a, u, slot, t, [&](int g, int d, Merge8& mg) {
    // kMergeBatch partials' loads in flight at a time: a long stream's last
    // segment merges ~76 of them, and each batch is one L2 round trip
    for (int k0 = 0; k0 < S; k0 += kMergeBatch) {
      float m[kMergeBatch], l[kMergeBatch], x[kMergeBatch][8];
#pragma unroll
      for (int q = 0; q < kMergeBatch; ++q) {
        const int k = k0 + q;
        m[q] = -INFINITY;
        l[q] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) x[q][i] = 0.f;
        if (cand_ok(k)) {
          const float* pk = a.part + static_cast<int64_t>(cand_slot(k)) * stride;
          m[q] = __ldcg(pk + GP * D + g);
          l[q] = __ldcg(pk + GP * D + GP + g);
          const float4 y0 = __ldcg(reinterpret_cast<const float4*>(pk + g * D + d));
          const float4 y1 = __ldcg(reinterpret_cast<const float4*>(pk + g * D + d + 4));
          x[q][0] = y0.x; x[q][1] = y0.y; x[q][2] = y0.z; x[q][3] = y0.w;
          x[q][4] = y1.x; x[q][5] = y1.y; x[q][6] = y1.z; x[q][7] = y1.w;
        }
      }
#pragma unroll
      for (int q = 0; q < kMergeBatch; ++q) mg.add(m[q], l[q], x[q]);
    }
  });
  if (t == 0) a.counters[u] = 0;
  team_sync<NTH>();
}

template <int D, int NT, bool PAGED, bool F8>
__global__ void __launch_bounds__(Geo<D, NT, F8>::THREADS, 1) decode_kernel(const __grid_constant__ DecodeArgs a) {
  using Gm = Geo<D, NT, F8>;
  constexpr int kWarps = Gm::W, kHelper = Gm::W, kThreads = Gm::THREADS;
  constexpr int GP = Gm::GP, KSTEPS = Gm::KSTEPS, BOXES = Gm::BOXES, KG = Gm::KG, NS = Gm::NS;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int warp_max[kThreads / 32];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const CacheView& c = a.c;
  const int Hkv = a.Hkv, U = a.B * Hkv;
  const int NC = gridDim.x, cta = blockIdx.x;
  int* P = reinterpret_cast<int*>(smem + Gm::TAB_OFF);  // [U + 1] tile prefix over units
  int* N = P + U + 1;                                    // [U] cached keys per unit
  int* HD = N + U;                                       // [U] ring: head slot
  int* RW = HD + U;                                      // [U] ring: cache row
  float* ML = reinterpret_cast<float*>(smem + Gm::ML_OFF);
  int* SLOT = reinterpret_cast<int*>(smem + Gm::SLOT_OFF);
  int* flag = reinterpret_cast<int*>(smem + Gm::FLAG_OFF);
  float2* cs = reinterpret_cast<float2*>(smem + Gm::CS_OFF);
  float* qs = reinterpret_cast<float*>(smem + Gm::QS_OFF);
  uint64_t* step = reinterpret_cast<uint64_t*>(smem + Gm::STEP_OFF);
  uint8_t* in_slots = smem + Gm::IN_OFF;
  const uint32_t stage_bars = smem_addr(smem + Gm::BAR_OFF);
  const uint32_t inbar = smem_addr(smem + Gm::INBAR_OFF);
  const uint32_t prep_full = smem_addr(smem + Gm::PREP_FULL_OFF);
  const uint32_t prep_empty = smem_addr(smem + Gm::PREP_EMPTY_OFF);
  const uint32_t merge_full = smem_addr(smem + Gm::MERGE_FULL_OFF);
  const uint32_t merge_empty = smem_addr(smem + Gm::MERGE_EMPTY_OFF);

  if (threadIdx.x == 32) {
    prefetch_tmap(&a.tmap_k);
    prefetch_tmap(&a.tmap_v);
  }
  if constexpr (PAGED) {
    // the page table into L2 (each CTA a share of its lines), for the window
    // fills that read it once the split is known
    const int64_t lines = (static_cast<int64_t>(a.B) * c.bt_stride + 31) / 32;
    if (lines <= kPrefetchLines)
      for (int64_t i = static_cast<int64_t>(cta) * kThreads + threadIdx.x; i < lines;
           i += static_cast<int64_t>(NC) * kThreads)
        prefetch_l2(c.block_table + i * 32);
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kWarps * NS; ++i) mbar_init(stage_bars + 8 * i, 1);
    mbar_init(inbar, 1);  // the input slots
    mbar_init(inbar + 8, 1);
    mbar_init(prep_full, 1);
    mbar_init(prep_empty, kWarps);
    mbar_init(merge_full, kWarps);
    mbar_init(merge_empty, 1);
    fence_mbar_init();
  }

  // ---- unit table: tiles per unit, then their prefix sum. A paged unit's
  // tiles follow from its length (caller metadata; no kernel of this library
  // writes it). A ring unit scans every 16-slot block of its ring, the valid
  // slots masked in when scored, so a ring layer's split needs none of its
  // metadata and its first copies go out before that metadata is read.
  const int ring_tiles = PAGED ? 0 : ((c.R + kGroup - 1) / kGroup + KG - 1) / KG;
  int max_tiles = 0;
  for (int u = threadIdx.x; u < U; u += kThreads) {
    int tiles = ring_tiles;
    if constexpr (PAGED) {
      const int b = u / Hkv;
      const int n = unit_length<true>(c, b, a.max_len, cta == 0 && u - b * Hkv == 0, a.err);
      N[u] = n;
      tiles = (paged_groups(c, n) + KG - 1) / KG;
    }
    P[u + 1] = tiles;
    max_tiles = max(max_tiles, tiles);
  }
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) max_tiles = max(max_tiles, __shfl_xor_sync(kFull, max_tiles, w));
  if (lane == 0) warp_max[warp] = max_tiles;
  if (threadIdx.x == 0) P[0] = 0;
  __syncthreads();
  block_scan_inclusive<kThreads>(P + 1, U);
  const int T = P[U];
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) max_tiles = max(max_tiles, warp_max[w]);

  // ---- the split of the tiles over the grid. Pieces: when there are no more
  // units than CTAs and cutting every unit into s = NC / U equal pieces (one
  // CTA each) leaves the largest piece within kPiecesSlack of a fair share,
  // CTA u * s + k takes piece k of unit u - units mostly end inside one CTA
  // and few partials cross CTAs. Otherwise stream-K over the units laid end to
  // end, each weighted with the fixed cost of a segment (Split).
  const Split sp{P, U, a.unit_cost, NC, T + static_cast<int64_t>(a.unit_cost) * U};
  int pieces = 0;
  if (U <= NC && T > 0) {
    const int s = NC / U;
    if (100 * ((max_tiles + s - 1) / s) <= (100 + kPiecesSlack) * ((T + NC - 1) / NC)) pieces = s;
  }
  int g0, g1;
  if (pieces) {
    const int u = cta / pieces, k = cta - u * pieces;
    const int t = u < U ? P[u + 1] - P[u] : 0;
    g0 = u < U ? P[u] + k * t / pieces : 0;
    g1 = u < U ? P[u] + (k + 1) * t / pieces : 0;
  } else {
    g0 = sp.tile_at(sp.bound(cta));
    g1 = sp.tile_at(sp.bound(cta + 1));
  }
  const int span = g1 - g0;
  // this CTA's units (segments), in order
  auto next_unit = [&](int u) {  // the next unit with tiles in this CTA's range
    for (++u; u < U && P[u] < g1; ++u)
      if (P[u + 1] > P[u]) return u;
    return U;
  };
  const int u_first = span > 0 ? unit_of(P, U, g0) : U;  // the first unit of a range has tiles in it
  int n_segs = 0, u_last = U;
  for (int u = u_first; u < U; u = next_unit(u)) {
    u_last = u;
    ++n_segs;
  }

  // Ordering with the preceding launch on the stream, which may still run:
  // it may be writing its new entries into its own cache, its outputs and its
  // partials (the other half of the double-buffered workspace). This call's
  // inputs, metadata and partials are never written by it. So the pass over
  // the cache runs before waiting for it when its cache is a different one
  // (a.early); the outputs and the write-back always come after the wait.
  // Each CTA waits before it lets the next launch begin, so at most two
  // calls are ever in flight.
  bool waited = false;
  auto wait_prev = [&]() {
    if (!waited) {
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
  };
  if (!a.early) wait_prev();

  if (warp != kHelper) {
    // ================= streaming warp: tiles g = g0 + warp + kWarps * it
    const int my_n = span > warp ? (span - warp + kWarps - 1) / kWarps : 0;
    uint8_t* wsm = smem + warp * NS * Gm::STAGE;
    const uint32_t wsm_a = smem_addr(wsm);
    const uint32_t bar0 = stage_bars + warp * NS * 8;
    int* wrow = reinterpret_cast<int*>(smem + Gm::WROW_OFF) + warp * 2 * kWin * KG;
    int* wmask = reinterpret_cast<int*>(smem + Gm::WMASK_OFF) + warp * 2 * kWin * KG;

    // Window w of this warp: tiles 32w..32w+31, one per lane. For each group of
    // the tile: the first tensor row of its TMA boxes and its valid-row mask
    // (0 = no such group). Stored in half (w & 1) of the warp's window arrays.
    auto fill = [&](int w) {
      const int x = w * kWin + lane;
      int rows[KG], masks[KG];
#pragma unroll
      for (int kg = 0; kg < KG; ++kg) rows[kg] = masks[kg] = 0;
      if (x < my_n) {
        const int g = g0 + warp + kWarps * x;
        const int u = unit_of(P, U, g);
        const int b = u / Hkv, j = u - b * Hkv;
        const int n = N[u];
        if constexpr (PAGED) {
          const int gpp = (c.P + kGroup - 1) / kGroup;
          const int groups = paged_groups(c, n);
#pragma unroll
          for (int kg = 0; kg < KG; ++kg) {
            const int gi = (g - P[u]) * KG + kg;
            if (gi < groups) {
              const int pi = gi / gpp, gr = gi - pi * gpp;
              int pg = c.block_table[static_cast<int64_t>(b) * c.bt_stride + pi];
              if (pg < 0 || pg >= c.n_rows) {
                raise_error(a.err, ERR_INDEX);
                pg = 0;
              }
              rows[kg] = (pg * Hkv + j) * c.P + gr * kGroup;
              masks[kg] = static_cast<int>(row_bits(0, min(c.P - gr * kGroup, n - (pi * c.P + gr * kGroup))));
            }
          }
        } else {
          // block gi of the ring: slots 16 gi .. 16 gi + 15, valid when they are
          // among the n slots before the head
          const int R = c.R, nb = (R + kGroup - 1) / kGroup;
          const int head = HD[u], row = RW[u];
          const int start = ring_start(head, n, R), end = start + n;  // valid: [start, end) mod R
#pragma unroll
          for (int kg = 0; kg < KG; ++kg) {
            const int gi = (g - P[u]) * KG + kg;
            if (gi < nb) {
              const int s0 = gi * kGroup;
              rows[kg] = (row * Hkv + j) * R + s0;
              uint32_t m = row_bits(start - s0, min(end, R) - s0);
              if (end > R) m |= row_bits(-s0, end - R - s0);
              masks[kg] = static_cast<int>(m);
            }
          }
        }
      }
      int* wr = wrow + (w & 1) * kWin * KG;
      int* wm = wmask + (w & 1) * kWin * KG;
#pragma unroll
      for (int kg = 0; kg < KG; ++kg) {
        wr[lane * KG + kg] = rows[kg];
        wm[lane * KG + kg] = masks[kg];
      }
      __syncwarp();
    };
    const uint64_t policy = l2_evict_first_policy();
    // Stages with copies in flight (bit st, kept by the issuing lane) and the
    // parity of each stage's next wait (bit 8 + st): a warp that gave up
    // waiting still lets its copies land before the CTA exits.
    uint32_t copies = 0;
    // The K and V rows of group kg of a stage from tensor row row0 on.
    auto load_group = [&](uint32_t kd, int kg, int row0, uint32_t bar) {
      if constexpr (kGroupBox<D> || F8) {
        // one box per group: 16 rows x every 128-byte region
        tma_load_3d(kd + kg * Gm::GBYTES, &a.tmap_k, 0, row0, 0, bar, policy);
        tma_load_3d(kd + Gm::KHALF + kg * Gm::GBYTES, &a.tmap_v, 0, row0, 0, bar, policy);
      } else {
        // one box per 64-dim region of the group
#pragma unroll
        for (int bx = 0; bx < BOXES; ++bx) {
          tma_load_2d(kd + kg * Gm::GBYTES + bx * kBoxBytes, &a.tmap_k, 64 * bx, row0, bar, policy);
          tma_load_2d(kd + Gm::KHALF + kg * Gm::GBYTES + bx * kBoxBytes, &a.tmap_v, 64 * bx, row0, bar, policy);
        }
      }
    };
    // Request tile x of this warp into stage x % NS (one lane): the groups
    // that hold a valid row.
    auto issue = [&](int x) {
      copies |= 1u << (x % NS);
      const int* wr = wrow + ((x / kWin) & 1) * kWin * KG + (x % kWin) * KG;
      const int* wm = wmask + ((x / kWin) & 1) * kWin * KG + (x % kWin) * KG;
      int gn = 0;
#pragma unroll
      for (int kg = 0; kg < KG; ++kg) gn += wm[kg] != 0;
      const uint32_t bar = bar0 + 8 * (x % NS);
      const uint32_t kd = wsm_a + (x % NS) * Gm::STAGE;
      mbar_arrive_expect_tx(bar, 2u * gn * Gm::GBYTES);
#pragma unroll
      for (int kg = 0; kg < KG; ++kg)
        if (wm[kg] != 0) load_group(kd, kg, wr[kg], bar);
    };
    const int pre = my_n < NS ? my_n : NS;
    if constexpr (!PAGED) {
      // A ring's first NS tiles go out from the split alone, every block of
      // them whole (the blocks past the ring's last slot are not requested);
      // which of their rows are valid is known by the time they are scored.
      // This thread's first unit's ring metadata is requested first, so that
      // its loads are in flight across the copies.
      const int um = threadIdx.x;  // (the streaming threads are 0 .. kWarps * 32 - 1)
      int m_row = 0, m_head = 0, m_cnt = 0;
      if (um < U) {
        const int b = um / Hkv;
        m_row = c.stream_rows ? c.stream_rows[b] : b;
        m_head = c.ring_head[b];
        m_cnt = c.ring_count[b];
      }
      // Lane x < NS works out tile x's first tensor row (its stream's cache
      // row loads for all tiles at once); lane 0 issues, once the helper warp
      // has requested the first units' inputs (their copies then go first).
      const int nb = (c.R + kGroup - 1) / kGroup;
      int row0 = 0, gi0 = 0;
      if (lane < pre) {
        const int g = g0 + warp + kWarps * lane;
        const int u = unit_of(P, U, g);
        const int b = u / Hkv, j = u - b * Hkv;
        int row = c.stream_rows ? c.stream_rows[b] : b;
        if (row < 0 || row >= c.n_rows) row = 0;  // (reported below; every slot is masked)
        gi0 = (g - P[u]) * KG;
        row0 = (row * Hkv + j) * c.R + gi0 * kGroup;
      }
      asm volatile("bar.sync 2, %0;" ::"r"(kThreads) : "memory");
      for (int x = 0; x < pre; ++x) {
        const int r0 = __shfl_sync(kFull, row0, x), b0 = __shfl_sync(kFull, gi0, x);
        if (lane == 0) {
          copies |= 1u << (x % NS);
          int gn = 0;
#pragma unroll
          for (int kg = 0; kg < KG; ++kg) gn += b0 + kg < nb;
          const uint32_t bar = bar0 + 8 * (x % NS);
          const uint32_t kd = wsm_a + (x % NS) * Gm::STAGE;
          mbar_arrive_expect_tx(bar, 2u * gn * Gm::GBYTES);
#pragma unroll
          for (int kg = 0; kg < KG; ++kg)
            if (b0 + kg < nb) load_group(kd, kg, r0 + kg * kGroup, bar);
        }
      }
      // then the ring metadata, shared out over the streaming warps (the only
      // readers: the windows' rows and masks)
      for (int u = um; u < U; u += kWarps * 32) {
        const int b = u / Hkv;
        int row = m_row, head = m_head, cnt = m_cnt;
        if (u != um) {
          row = c.stream_rows ? c.stream_rows[b] : b;
          head = c.ring_head[b];
          cnt = c.ring_count[b];
        }
        const int n = ring_length(c, row, head, cnt, cta == 0 && u - b * Hkv == 0, a.err);
        HD[u] = n > 0 ? head : 0;
        RW[u] = row;
        N[u] = n;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(kWarps * 32) : "memory");
    }
    fill(0);  // window 1 is filled once the first tiles are requested
    if (PAGED && lane == 0)
      for (int x = 0; x < pre; ++x) issue(x);

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
    // heads of this lane's score / output columns (e = 0, 1): the hi and lo
    // columns of one head are lanes l and l ^ 2 (NT == 1) or tiles 0 and 1 (NT == 2)
    const int hbase = NT == 1 ? 2 * (lane & 1) : fc;
    const bool lo_lane = NT == 1 && (lane & 2) != 0;

    bool failed = false;
    auto check = [&](bool ok) {  // the whole warp agrees, so its collectives stay converged
      if (!failed && !__all_sync(kFull, ok)) {
        failed = true;
        if (lane == 0) raise_error(a.err, ERR_TIMEOUT);
      }
    };
    int it = 0;
    int held = -1;  // tile whose stage still holds the previous segment's merge buffer
    int seg = 0;
    for (int u = u_first; u < U; u = next_unit(u), ++seg) {
      const int ge = min(g1, P[u + 1]);

      // ---- the unit's rotated q from the helper, as B fragments: column n =
      // fg of tile t holds one head's hi or lo part
      if (!failed) check(mbar_wait_bounded(prep_full, seg & 1, a.wait_ns));
      uint32_t qb[KSTEPS][NT][2];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int head = NT == 1 ? (fg & 3) : fg;
        const bool lo = NT == 1 ? fg >= 4 : t == 1;
        const float* src = qs + head * D;
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            // bf16 K: the fragment's k-pairs are dims 2c, 2c + 8 of the step
            // (c = lane % 4); E4M3 K: dims 4c and 4c + 2 (the order its bytes
            // reach the A fragment, applied to both operands alike)
            const int dim = F8 ? ks * 16 + 4 * (lane & 3) + 2 * h2 : ks * 16 + fc + 8 * h2;
            const float2 x = *reinterpret_cast<const float2*>(src + dim);
            uint32_t hi, lw;
            if constexpr (F8)
              split_f16x2(x.x, x.y, hi, lw);
            else
              split_bf16x2(x.x, x.y, hi, lw);
            qb[ks][t][h2] = lo ? lw : hi;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(prep_empty);

      float o[KSTEPS][NT][4];
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[mt][t][e] = 0.f;
      float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
      int last_stage = -1, pend = -1;

      for (;;) {
        const int g = g0 + warp + kWarps * it;
        if (it >= my_n || g >= ge) break;
        // the next window: its half was last read for tiles now behind
        if ((it & (kWin - 1)) == 0 && it + kWin < my_n) fill(it / kWin + 1);
        // the previous segment's merge buffer streams again once the helper has read it
        if (held >= 0) {
          bool ready;
          if (held == it) {
            if (!failed) check(mbar_wait_bounded(merge_empty, (seg - 1) & 1, a.wait_ns));
            ready = true;
          } else {
            ready = __shfl_sync(kFull, mbar_test_wait(merge_empty, (seg - 1) & 1) ? 1 : 0, 0) != 0;
          }
          if (ready) {
            if (lane == 0 && !failed) issue(held);
            held = -1;
          }
        }
        const int stg = it % NS;
        if (!failed) {
          check(mbar_wait_bounded(bar0 + 8 * stg, (it / NS) & 1, a.wait_ns));
          copies &= ~(1u << stg);
          copies ^= 0x100u << stg;
        }
        if (!failed) {
          const int* wm = wmask + ((it / kWin) & 1) * kWin * KG + (it % kWin) * KG;
#pragma unroll
          for (int kg = 0; kg < KG; ++kg) {
            const uint32_t mask = static_cast<uint32_t>(wm[kg]);
            if (mask == 0u) continue;  // no valid row (past a unit's end, or a ring's unwritten block)
            const uint32_t kbase = wsm_a + stg * Gm::STAGE + kg * Gm::GBYTES;
            const uint32_t vbase = kbase + Gm::KHALF;
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
            if constexpr (F8) {
              // 32 bytes of 16 rows per load: E4M3 dims 4c..4c+3 of rows r and
              // r + 8 (and 16 dims on), widened exactly to fp16 pairs: two k-steps
#pragma unroll
              for (int j = 0; j < KSTEPS / 2; ++j) {
                uint32_t af[4];
                ldsm_x4(kbase + (j >> 2) * kBoxBytes + koff[j & 3], af);
                const uint32_t a0[4] = {e4m3x2_lo(af[0]), e4m3x2_lo(af[1]), e4m3x2_hi(af[0]), e4m3x2_hi(af[1])};
                const uint32_t a1[4] = {e4m3x2_lo(af[2]), e4m3x2_lo(af[3]), e4m3x2_hi(af[2]), e4m3x2_hi(af[3])};
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                  mma_f16(sacc[0][t], a0, qb[2 * j][t][0], qb[2 * j][t][1]);
                  mma_f16(sacc[1][t], a1, qb[2 * j + 1][t][0], qb[2 * j + 1][t][1]);
                }
              }
            } else {
#pragma unroll
              for (int ks = 0; ks < KSTEPS; ++ks) {
                uint32_t af[4];
                ldsm_x4(kbase + (ks >> 2) * kBoxBytes + koff[ks & 3], af);
#pragma unroll
                for (int t = 0; t < NT; ++t) mma_bf16(sacc[ks & 1][t], af, qb[ks][t][0], qb[ks][t][1]);
              }
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
              if constexpr (F8) {
                split_f16x2(p[0], p[1], h01, l01);
                split_f16x2(p[2], p[3], h23, l23);
              } else {
                split_bf16x2(p[0], p[1], h01, l01);
                split_bf16x2(p[2], p[3], h23, l23);
              }
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
            if constexpr (F8) {
              // V^T from E4M3 rows: the transposing load of 16 keys x 32 bytes
              // (the bf16 path's offsets) gives each lane, per 8x8 b16 matrix,
              // dims 2f, 2f + 1 (f = lane / 4) of keys 2c, 2c + 1 (c = lane % 4);
              // one byte permute makes key pairs per dim, widened exactly to
              // fp16. The A rows of m-tile mt are dims 16 mt + 2f (row f) and
              // 16 mt + 2f + 1 (row f + 8); the outputs are put back in order
              // when stored.
#pragma unroll
              for (int pj = 0; pj < KSTEPS / 2; ++pj) {
                uint32_t af[4];
                ldsm_x4_t(vbase + (pj >> 2) * kBoxBytes + voff[pj & 3], af);
                uint32_t kp[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) kp[x] = prmt(af[x], 0u, 0x3120u);
                // matrices: 0 = keys 0-7 / dims 0-15, 1 = keys 0-7 / dims 16-31,
                // 2 = keys 8-15 / dims 0-15, 3 = keys 8-15 / dims 16-31
                const uint32_t a0[4] = {e4m3x2_lo(kp[0]), e4m3x2_hi(kp[0]), e4m3x2_lo(kp[2]), e4m3x2_hi(kp[2])};
                const uint32_t a1[4] = {e4m3x2_lo(kp[1]), e4m3x2_hi(kp[1]), e4m3x2_lo(kp[3]), e4m3x2_hi(kp[3])};
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                  mma_f16(o[2 * pj][t], a0, pb[t][0], pb[t][1]);
                  mma_f16(o[2 * pj + 1][t], a1, pb[t][0], pb[t][1]);
                }
              }
            } else {
#pragma unroll
              for (int mt = 0; mt < KSTEPS; ++mt) {
                uint32_t af[4];
                ldsm_x4_t(vbase + (mt >> 2) * kBoxBytes + voff[mt & 3], af);
#pragma unroll
                for (int t = 0; t < NT; ++t) mma_bf16(o[mt][t], af, pb[t][0], pb[t][1]);
              }
            }
          }
          __syncwarp();
        }

        last_stage = stg;
        // Refill this stage with the warp's tile NS ahead. The warp's last tile
        // of a segment keeps its stage as the merge buffer until the helper
        // (or the CTA) has read it.
        if (it + NS < my_n) {
          if (g + kWarps >= ge) {
            pend = it + NS;
          } else if (lane == 0 && !failed) {
            issue(it + NS);
          }
        }
        ++it;
      }

      // ---- this warp's state: l summed over the lanes of a head, O^T to the
      // merge buffer as o[head][dim] (hi + lo columns). The previous
      // segment's buffers must have been read first (ML and SLOT are reused).
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        l_run[e] += __shfl_xor_sync(kFull, l_run[e], 4);
        l_run[e] += __shfl_xor_sync(kFull, l_run[e], 8);
        l_run[e] += __shfl_xor_sync(kFull, l_run[e], 16);
      }
      if (seg > 0) {
        if (!failed) check(mbar_wait_bounded(merge_empty, (seg - 1) & 1, a.wait_ns));
        if (held >= 0) {
          if (lane == 0 && !failed) issue(held);
          held = -1;
        }
      }
      held = pend;
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
            // (E4M3 V: its m-tiles hold permuted dims, and its values its scale)
            const int dim = F8 ? mt * 16 + 2 * fg + (i >> 1) : mt * 16 + fg + 8 * (i >> 1);
            if (writer) os[(hbase + (i & 1)) * D + dim] = F8 ? v * a.v_scale : v;
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
      __syncwarp();
      if (lane == 0) mbar_arrive(merge_full);
    }
    // copies still in flight exist only after a wait gave up: let them land
    if (lane == 0)
      for (int st = 0; st < NS; ++st)
        if ((copies >> st) & 1u) mbar_wait_bounded(bar0 + 8 * st, (copies >> (8 + st)) & 1u, a.wait_ns);
    __syncwarp();
  } else {
    // ================= helper warp: the units' inputs, RoPE and new token one
    // segment ahead; the end of every segment but the CTA's last
    bool failed = false;
    auto check = [&](bool ok) {
      if (!failed && !__all_sync(kFull, ok)) {
        failed = true;
        if (lane == 0) raise_error(a.err, ERR_TIMEOUT);
      }
    };
    int n_st = 0;  // units staged so far; unit k of this CTA uses input slot k & 1
    int pos_s[2] = {0, 0}, unit_s[2] = {0, 0};
    uint16_t gate_s[2] = {0, 0};  // raw bf16: converting here would wait for the load
    auto stage = [&](int u) {
      const int b = u / Hkv, j = u - b * Hkv, sl = n_st & 1;
      __syncwarp();  // every lane's reads of the slot come first
      if (lane == 0) issue_stage<D, GP>(a, u, n_st, inbar, in_slots, step);
      const int pv = a.pos[b];
      const uint16_t gv = (a.gate && lane < a.G) ? a.gate[(static_cast<int64_t>(b) * Hkv + j) * a.G + lane] : 0;
      if (sl == 0) {
        pos_s[0] = pv;
        gate_s[0] = gv;
        unit_s[0] = u;
      } else {
        pos_s[1] = pv;
        gate_s[1] = gv;
        unit_s[1] = u;
      }
      ++n_st;
    };
    // rotated q of the CTA's k-th unit into qs (then PREP_FULL), its new token into its slot
    auto prep = [&](int k) {
      const int sl = k & 1;
      if (!failed) check(mbar_wait_bounded(inbar + 8 * sl, (k >> 1) & 1, a.wait_ns));
      uint8_t* slot = in_slots + sl * Gm::IN_BYTES;
      if (a.q_norm || a.k_norm)
        norm_staged<D, 32>(a, reinterpret_cast<uint16_t*>(slot + Gm::IN_Q),
                           reinterpret_cast<uint16_t*>(slot + Gm::IN_K), lane);
      prep_q<D, GP, 32>(a, reinterpret_cast<const uint16_t*>(slot + Gm::IN_Q), sl ? pos_s[1] : pos_s[0], step,
                        qs, cs, lane);
      __syncwarp();
      // (a testing aid can withhold the first unit's q, so that every
      // streaming warp's bounded wait for it runs out)
      if (lane == 0 && !(k == 0 && (a.debug_flags & kDebugWithholdQ))) mbar_arrive(prep_full);
      // the new entry's target, read once the unit's segments are done: its
      // metadata loads are off the CTA's tail (prep_token ends with a barrier)
      if (a.write_back && lane == 0) {
        const int uk = sl ? unit_s[1] : unit_s[0];
        *reinterpret_cast<int64_t*>(slot + Gm::IN_WB) = write_back_offset<PAGED>(a, uk / Hkv, uk % Hkv, D);
      }
      prep_token<D, GP, 32>(a, qs, cs, slot, sl ? gate_s[1] : gate_s[0], lane);
    };
    if (u_first < U) {
      stage(u_first);
      const int u1 = next_unit(u_first);
      if (u1 < U) stage(u1);
    }
    // (a ring layer's streaming warps issue their first copies after this)
    if constexpr (!PAGED) asm volatile("bar.arrive 2, %0;" ::"r"(kThreads) : "memory");
    if (u_first < U) prep(0);
    int seg = 0;
    for (int u = u_first; u < U; ++seg) {
      const int un = next_unit(u);
      if (un >= U) break;  // the CTA's last segment is ended by the whole CTA
      // the next unit's q, once every streaming warp has read this one's
      if (!failed) check(mbar_wait_bounded(prep_empty, seg & 1, a.wait_ns));
      prep(seg + 1);
      // this segment's end
      if (!failed) check(mbar_wait_bounded(merge_full, seg & 1, a.wait_ns));
      end_segment<D, NT, PAGED, F8, 32>(a, sp, pieces, u, seg == 0, cta, smem, ML, SLOT,
                                    in_slots + (seg & 1) * Gm::IN_BYTES, flag, lane, wait_prev, [&] {
                                      fence_proxy_async_smem();
                                      __syncwarp();
                                      if (lane == 0) mbar_arrive(merge_empty);
                                    });
      // its slot is free: the unit after next
      const int unn = next_unit(un);
      if (unn < U) stage(unn);
      u = un;
    }
  }

  // ---- the CTA's last segment, ended by all threads
  __syncthreads();
  if (u_last < U) {
    const int sl = n_segs - 1;
    end_segment<D, NT, PAGED, F8, kThreads>(a, sp, pieces, u_last, sl == 0, cta, smem, ML, SLOT,
                                        in_slots + (sl & 1) * Gm::IN_BYTES, flag, threadIdx.x, wait_prev, [] {});
  }

  // ---- units with no cached keys have no segments: CTA u % NC finishes them
  int n = n_segs;
  for (int u = cta; u < U; u += NC) {
    if (P[u + 1] != P[u]) continue;
    __syncthreads();  // the slot, qs and cs may still be read
    const int b = u / Hkv, j = u - b * Hkv;
    if (threadIdx.x == 0) issue_stage<D, GP>(a, u, n, inbar, in_slots, step);
    const int pos = a.pos[b];
    const uint16_t gr =
        (a.gate && threadIdx.x < a.G) ? a.gate[(static_cast<int64_t>(b) * Hkv + j) * a.G + threadIdx.x] : 0;
    if (!mbar_wait_bounded(inbar + 8 * (n & 1), (n >> 1) & 1, a.wait_ns)) raise_error(a.err, ERR_TIMEOUT);
    uint8_t* slot = in_slots + (n & 1) * Gm::IN_BYTES;
    if (a.q_norm || a.k_norm)
      norm_staged<D, kThreads>(a, reinterpret_cast<uint16_t*>(slot + Gm::IN_Q),
                               reinterpret_cast<uint16_t*>(slot + Gm::IN_K), threadIdx.x);
    prep_q<D, GP, kThreads>(a, reinterpret_cast<const uint16_t*>(slot + Gm::IN_Q), pos, step, qs, cs, threadIdx.x);
    if (a.write_back && threadIdx.x == 0)
      *reinterpret_cast<int64_t*>(slot + Gm::IN_WB) = write_back_offset<PAGED>(a, b, j, D);
    __syncthreads();
    prep_token<D, GP, kThreads>(a, qs, cs, slot, gr, threadIdx.x);
    wait_prev();
    finish_unit<D, GP, PAGED, kThreads>(a, u, slot, threadIdx.x, [](int, int, Merge8&) {});
    ++n;
  }
  wait_prev();
}

// ---------------------------------------------------------------- launch

template <int D, int NT, bool PAGED, bool F8>
cudaError_t decode_launch(const DecodeArgs& a, int ctas, cudaStream_t s, bool pdl) {
  using Gm = Geo<D, NT, F8>;
  auto k = decode_kernel<D, NT, PAGED, F8>;
  static std::atomic<uint64_t> opted{0};
  const cudaError_t e = opt_in_smem(k, Gm::SMEM_MAX, opted);
  if (e != cudaSuccess) return e;
  const size_t smem = 1024 + Gm::TAB_OFF + (4 * a.B * a.Hkv + 1) * sizeof(int);
  if (!pdl) {
    k<<<ctas, Gm::THREADS, smem, s>>>(a);
    return cudaGetLastError();
  }
  return launch_pdl(k, dim3(ctas), dim3(Gm::THREADS), smem, s, a);
}

template <int D, int NT, bool F8>
cudaError_t decode_dispatch_paged(const DecodeArgs& a, int ctas, cudaStream_t s, bool pdl) {
  return a.c.paged ? decode_launch<D, NT, true, F8>(a, ctas, s, pdl) : decode_launch<D, NT, false, F8>(a, ctas, s, pdl);
}

template <bool F8>
cudaError_t decode_dispatch(const DecodeArgs& a, int D, int GP, int ctas, cudaStream_t s, bool pdl) {
  if (D == 256) {
    if (GP == 4) return decode_dispatch_paged<256, 1, F8>(a, ctas, s, pdl);
    if (GP == 8) return decode_dispatch_paged<256, 2, F8>(a, ctas, s, pdl);
  } else if (D == 128) {
    if (GP == 4) return decode_dispatch_paged<128, 1, F8>(a, ctas, s, pdl);
    if (GP == 8) return decode_dispatch_paged<128, 2, F8>(a, ctas, s, pdl);
  }
  return cudaErrorNotSupported;
}

}  // namespace

#ifdef DATTN_DECODE_FP8_UNIT
// This translation unit holds the E4M3-cache instantiations only (compiled
// beside the bf16 ones, in parallel).
cudaError_t launch_decode_fp8(const DecodeArgs& a, int D, int GP, int ctas, cudaStream_t s, bool pdl) {
  return decode_dispatch<true>(a, D, GP, ctas, s, pdl);
}
#else
namespace {

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

cudaError_t encode_cache_maps(const CacheView& c, int Hkv, int D, CUtensorMap* k, CUtensorMap* v, bool f8) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn) return cudaErrorNotSupported;
  const uint64_t rows = static_cast<uint64_t>(c.n_rows) * Hkv * (c.paged ? c.P : c.R);
  if (rows == 0 || rows > 0x7fffffffull) return cudaErrorNotSupported;
  if (f8) {
    // E4M3 rows of D bytes: a 3D view (128 bytes, row, D/128 regions), one
    // box per 16-row group, 128-byte swizzled like the bf16 groups
    const cuuint64_t dims[3] = {128, rows, static_cast<cuuint64_t>(D / 128)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D), 128};
    const cuuint32_t box[3] = {128, kGroup, static_cast<cuuint32_t>(D / 128)};
    const cuuint32_t estride[3] = {1, 1, 1};
    for (int i = 0; i < 2; ++i) {
      const CUresult r = fn(i ? v : k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, i ? c.v : c.k, dims, strides, box,
                            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    return cudaSuccess;
  }
  // D = 128: a 3D view of the [rows, D] bf16 cache, (64 dims, row, 64-dim
  // region), so that one box brings a 16-row group as its regions of 16 rows x
  // 128 bytes one after the other; D = 256: the 2D [rows, D] view, one box
  // per region. Either way the 128-byte-swizzled layout the MMAs read.
  const bool group_box = D == 128 ? kGroupBox<128> : kGroupBox<256>;
  const cuuint32_t rank = group_box ? 3 : 2;
  const cuuint64_t dims[3] = {group_box ? 64u : static_cast<cuuint64_t>(D), rows,
                              static_cast<cuuint64_t>(D / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, 128};
  const cuuint32_t box[3] = {64, kGroup, static_cast<cuuint32_t>(D / 64)};
  const cuuint32_t estride[3] = {1, 1, 1};
  for (int i = 0; i < 2; ++i) {
    const CUresult r = fn(i ? v : k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, i ? c.v : c.k, dims, strides,
                          box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

cudaError_t encode_verify_maps(const CacheView& c, int Hkv, int D, const uint16_t* qhl, int qhl_rows, int Hq,
                               int G, int S, int T, CUtensorMap* k, CUtensorMap* v, CUtensorMap* q) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn) return cudaErrorNotSupported;
  const uint64_t rows = static_cast<uint64_t>(c.n_rows) * Hkv * (c.paged ? c.P : c.R);
  if (rows == 0 || rows > 0x7fffffffull) return cudaErrorNotSupported;
  {
    // K: 2D [rows, D], one box = 16 rows x 64 dims
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
    const cuuint32_t box[2] = {64, kGroup};
    const cuuint32_t estride[2] = {1, 1};
    const CUresult r = fn(k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c.k, dims, strides, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  {
    // V: 3D (64 dims, row, 64-dim region), one box = a 16-row group, every region
    const cuuint64_t dims[3] = {64, rows, static_cast<cuuint64_t>(D / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, 128};
    const cuuint32_t box[3] = {64, kGroup, static_cast<cuuint32_t>(D / 64)};
    const cuuint32_t estride[3] = {1, 1, 1};
    const CUresult r = fn(v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, c.v, dims, strides, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq),
                              static_cast<cuuint64_t>(S) * T, 2};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hq) * D * 2,
                                 static_cast<cuuint64_t>(qhl_rows) * Hq * D * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(T), 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  const CUresult r = fn(q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(qhl), dims, strides, box,
                        estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_decode(const DecodeArgs& args, int D, int ctas, cudaStream_t s, bool pdl) {
  DecodeArgs a = args;
  a.unit_cost = kSegmentCost;
  if (a.wait_ns == 0) a.wait_ns = kDefaultWaitNs;
  const int GP = decode_group_pad(a.G);
  if (a.B * a.Hkv > kMaxUnits) return cudaErrorNotSupported;
  if (a.r > D || a.r % 2 != 0) return cudaErrorNotSupported;
  if (a.f8) return launch_decode_fp8(a, D, GP, ctas, s, pdl);
  return decode_dispatch<false>(a, D, GP, ctas, s, pdl);
}

// Keys of one round of stage tiles over the streaming warps, in units of 4
// tiles (the grid plan gives each CTA at least one round).
int decode_tile_keys(int D, int G, bool f8) {
  const int GP = decode_group_pad(G);
  if (GP == 0 || (D != 128 && D != 256)) return 0;
  auto keys = [](int kg, int w) { return kGroup * kg * w / 4; };
  if (D == 256) {
    if (f8) return GP == 4 ? keys(Geo<256, 1, true>::KG, Geo<256, 1, true>::W) : keys(Geo<256, 2, true>::KG, Geo<256, 2, true>::W);
    return GP == 4 ? keys(Geo<256, 1>::KG, Geo<256, 1>::W) : keys(Geo<256, 2>::KG, Geo<256, 2>::W);
  }
  if (f8) return GP == 4 ? keys(Geo<128, 1, true>::KG, Geo<128, 1, true>::W) : keys(Geo<128, 2, true>::KG, Geo<128, 2, true>::W);
  return GP == 4 ? keys(Geo<128, 1>::KG, Geo<128, 1>::W) : keys(Geo<128, 2>::KG, Geo<128, 2>::W);
}

int decode_ctas_per_sm(int D, int G) {
  const int GP = decode_group_pad(G);
  int smem = 0;
  // (the larger of the bf16 and E4M3 layouts: an E4M3 tile holds more groups)
  const auto larger = [](int x, int y) { return x > y ? x : y; };
  if (D == 256)
    smem = GP == 4   ? larger(Geo<256, 1>::SMEM_MAX, Geo<256, 1, true>::SMEM_MAX)
           : GP == 8 ? larger(Geo<256, 2>::SMEM_MAX, Geo<256, 2, true>::SMEM_MAX)
                     : 0;
  if (D == 128)
    smem = GP == 4   ? larger(Geo<128, 1>::SMEM_MAX, Geo<128, 1, true>::SMEM_MAX)
           : GP == 8 ? larger(Geo<128, 2>::SMEM_MAX, Geo<128, 2, true>::SMEM_MAX)
                     : 0;
  if (smem == 0) return 0;
  // 228 KB of shared memory per SM; 1 KB reserved and the static block-scan scratch per CTA
  const int per_sm = 233472 / (smem + 1024 + 64);
  return per_sm > 2 ? 2 : per_sm;
}

int decode_max_units() { return kMaxUnits; }
#endif  // DATTN_DECODE_FP8_UNIT

}  // namespace dattn
