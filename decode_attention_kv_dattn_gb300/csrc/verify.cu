// Tree verify: S streams x T draft rows, each row under its own tree mask
// ("TensorFold PR #608": verify rounds take every stream's window together, up
// to 16 streams of 16 rows). Row i of stream s sits at position
// prefix_len + depth(i) and attends to the stream's whole paged prefix, its
// ancestors in the tree and itself.
//
// Three launches, each a programmatic dependent of the one before:
//  * rope_kernel (rope.cu) - every row's q rotated (fp32 for the combine, and
//    as two bf16 terms hi + lo for the tensor-core pass) and the window keys'
//    bf16 entries.
//  * verify_split_kernel - the prefix, on the 5th-generation tensor cores. The
//    G*T rows of one (stream, KV head) unit share every prefix key, so a unit
//    is one 128-row MMA tile, and the keys come 128 per tile:
//        S (rows x 128 keys) = q_hi K^T + q_lo K^T     (bf16; q_hi in TMEM,
//                                                       q_lo in shared memory)
//        O (rows x D)       += P V                     (fp16; P in shared memory)
//    K enters exactly as it is stored (bf16) and q keeps 16 significant bits
//    as two bf16 terms: one rounding of q to 8 or 11 bits breaks the tolerance
//    once the softmax is peaked. Each softmax thread owns
//    one row (one TMEM lane): its running maximum, the lazy rescale of its
//    output row (only when the tile maximum passes the reference by more than
//    2^8, base 2) and its row sum stay in the thread. The scores leave tensor
//    memory as soon as the softmax threads hold them, so the next tile's
//    Q K^T runs while this tile's probabilities are formed.
//    Loads: the TMA unit lands K by tensor-map boxes of 16 keys x 64 dims
//    into a ring of 64-dim tile regions, and V by one box per 16-key page
//    group (all dims) into a ring of page-group slots, 128-byte swizzled, in
//    the order the MMAs consume them. K is used as it lands; four converter
//    warps turn each V slot from bf16 into fp16 in place (exact below 65504 in
//    magnitude, which they check: P is fp16, and bf16 probabilities would
//    break the tolerance) and zero the V rows of keys outside the prefix
//    (their probability is 0, but 0 x NaN is NaN). The q_lo and P operand
//    regions hold only the rows in use, which leaves the rings the room to
//    keep a tile in flight behind the one being consumed. Work is split
//    stream-K over all units' 128-key tiles.
//  * verify_combine_kernel - per (stream, row, KV head): merges the prefix
//    segments, scores the row's tree path in fp32 and joins it in score
//    space, applies the gate, stores fp32 and writes the window entries back.
#include <cuda_fp16.h>

#include "common.cuh"
#include "mma.cuh"
#include "tc.cuh"

namespace dattn {

namespace {

constexpr int KT = 128;                    // keys per tile: the Q K^T MMAs' N
constexpr int VM = 128;                    // MMA rows (G*T <= VM)
constexpr int kKChunk = 16384;             // bytes of one K ring slot: one 64-dim region of a tile
constexpr int kMaxK = 8;                   // K ring slots
constexpr int kKExtra = 0;                 // K slots beyond one tile's regions, when they fit
constexpr int kMaxV = 24;                  // V ring slots: one 16-key page group (all dims) each
constexpr int kSoftWarps = 8;              // warps 0..7: TMEM lane quarter w % 4 (one row per
                                           // lane), keys [64 (w / 4), 64 (w / 4) + 64) of the tile
constexpr int kTmaWarp = 8;                // issues the K and q_lo TMA copies
constexpr int kMmaWarp = 9;                // issues the Q K^T MMAs (one thread); owns TMEM
constexpr int kConv0 = 10, kConvWarps = 4; // V: bf16 -> fp16 in place
constexpr int kTmaVWarp = 14;              // issues the V TMA copies
constexpr int kPvWarp = 15;                // issues the P V MMAs (one thread)
constexpr int kVThreads = (kPvWarp + 1) * 32;
constexpr float kRescaleLog2 = 8.f;        // lazy rescale threshold (base 2)
constexpr int kTileRing = 8;               // tiles whose group rows and masks are kept
constexpr int kSmemLimit = 232448 - 64;    // dynamic shared memory per CTA (the static block-scan
                                           // scratch, 48 bytes, takes from the same 227 KB)
static_assert(kVerifyTileKeys == KT, "tile size shared with the host split");

// barrier indices
enum {
  B_KFULL = 0,                 // [kMaxK] K slot landed (TMA transaction bytes)
  B_KFREE = kMaxK,             // [kMaxK] the Q K^T MMAs reading the K slot completed
  B_VFULL = 2 * kMaxK,         // [kMaxV] V slot landed
  B_VCONV = 2 * kMaxK + kMaxV, // [kMaxV] V slot converted (one arrival per converter warp)
  B_VFREE = 2 * kMaxK + 2 * kMaxV,  // [kMaxV] the P V MMA reading the V slot completed
  B_QLO = 2 * kMaxK + 3 * kMaxV,    // the segment's q_lo rows landed in shared memory
  B_QHI,                       // the segment's q_hi rows are in TMEM (softmax warps)
  B_QFREE,                     // the segment's Q K^T MMAs completed (q may be replaced)
  B_SFULL,                     // Q K^T of the tile completed
  B_SFREE,                     // the softmax warps hold the tile's scores (S may be rewritten)
  B_PFULL,                     // P of the tile written to shared memory (softmax warps)
  B_PVDONE,                    // P V of the tile completed (P and O free)
  B_OFREE,                     // the segment's output has been read out of TMEM
  B_FINAL,                     // every MMA of the CTA completed (before TMEM is freed)
  B_COUNT
};

// A partial row is o[D], m, l, padded to a 16-byte multiple: D + 4 floats.
template <int D>
constexpr int row_stride() { return D + 4; }

// Shared-memory layout of one CTA for U units of R rows; the host computes the
// same to size the launch. An MMA operand region (64 dims or 64 keys of every
// row, 128 B per row) holds only the R rows rounded up to a core group of 8;
// the M = 128 MMAs read rows past that from whatever follows, and those rows'
// results are never used.
struct VLayout {
  int rb;        // bytes of one operand region: 128 * round8(R)
  int qlo_off;   // q_lo (A of the second Q K^T MMA): [D/64 regions][rows][128 B]
  int p_off;     // P (A of P V): [2 key regions of 64][rows][128 B]
  int ring_off;  // the K ring (ck slots of kKChunk), then the V ring (cv slots of 32 D bytes)
  int ck, cv;
  int bar_off;
  int misc_off;  // 32 bytes: tmem base (+0), the abort flag (+16)
  int xch_off;   // float XMAX[2 tile parities][2 halves][128], XL[2 halves][128]: the two key
                 // halves of a row meet here
  int trow_off;  // int TROW[kTileRing][8], TMASK[kTileRing][8], VMASK[kTileRing][8]
  int tab_off;   // int PT[U + 1], NK[U]
  int total;     // bytes, plus 1024 for the alignment of the base
};

__host__ __device__ inline VLayout verify_layout(int D, int U, int R) {
  VLayout L;
  L.rb = ((R + 7) / 8) * 1024;
  L.qlo_off = 0;
  L.p_off = (D / 64) * L.rb;
  L.ring_off = L.p_off + (KT / 64) * L.rb;
  const int tail = B_COUNT * 8 + 32 + 6 * 128 * 4 + 3 * kTileRing * 8 * 4 + (2 * U + 1) * 4;
  const int room = kSmemLimit - 1024 - L.ring_off - tail;
  // The K ring holds at least a whole tile's K (D/64 slots): its copy warp
  // issues a new segment's q_lo rows only after that segment's first K tile,
  // whose Q K^T needs them. The V ring takes the rest.
  L.ck = D / 64 + kKExtra;
  if ((room - L.ck * kKChunk) / (32 * D) < 8) L.ck = D / 64;
  L.cv = (room - L.ck * kKChunk) / (32 * D);
  if (L.cv > kMaxV) L.cv = kMaxV;
  L.bar_off = L.ring_off + L.ck * kKChunk + L.cv * 32 * D;
  L.misc_off = L.bar_off + B_COUNT * 8;
  L.xch_off = L.misc_off + 32;
  L.trow_off = L.xch_off + 6 * 128 * 4;
  L.tab_off = L.trow_off + 3 * kTileRing * 8 * 4;
  L.total = L.tab_off + (2 * U + 1) * 4 + 1024;
  return L;
}

// TMEM columns: q_hi (D/2 columns of bf16 pairs, the A operand of Q K^T), the
// scores of a tile (128), the output (D).
template <int D>
struct VCols {
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t S = D / 2;
  static constexpr uint32_t O = D / 2 + KT;
  static constexpr uint32_t TOTAL = D / 2 + KT + D;  // 512 at D = 256, 320 at 128
};

struct Waiter {
  uint32_t bars;
  volatile int* abort;
  int* err;
  // Bounded wait; on a timeout (or when another role gave up) every role
  // leaves its loop and the CTA frees its tensor memory.
  __device__ __forceinline__ bool wait(int b, uint32_t parity) const {
    const uint32_t bar = bars + 8 * b;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
      for (int i = 0; i < 32; ++i)
        if (mbar_try_wait(bar, parity)) return true;
      if (*abort) return false;
      if (global_timer_ns() - t0 > kDefaultWaitNs) {
        *abort = 1;
        raise_error(err, ERR_TIMEOUT);
        return false;
      }
    }
  }
};

__device__ __forceinline__ uint32_t cvt_pair_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// 16 bytes of 8 bf16 values turned into 8 fp16 values in place (exact below
// 65504 in magnitude); `mag` keeps the largest magnitude seen per 16-bit half.
__device__ __forceinline__ void convert16(uint8_t* p, uint32_t& mag) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  mag = __vmaxu2(mag, w.x & 0x7fff7fffu);
  mag = __vmaxu2(mag, w.y & 0x7fff7fffu);
  mag = __vmaxu2(mag, w.z & 0x7fff7fffu);
  mag = __vmaxu2(mag, w.w & 0x7fff7fffu);
  *reinterpret_cast<uint4*>(p) =
      make_uint4(cvt_pair_f16(bf16_lo(w.x), bf16_hi(w.x)), cvt_pair_f16(bf16_lo(w.y), bf16_hi(w.y)),
                 cvt_pair_f16(bf16_lo(w.z), bf16_hi(w.z)), cvt_pair_f16(bf16_lo(w.w), bf16_hi(w.w)));
}

template <int D>
__global__ void __launch_bounds__(kVThreads, 1) verify_split_kernel(const __grid_constant__ VerifySplitArgs a) {
  constexpr int NREG = D / 64;        // 64-dim regions: K chunks per tile
  constexpr int VG = 32 * D;          // bytes of one V slot: 16 keys x D dims
  using Col = VCols<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const CacheView& c = a.c;
  const int Hkv = a.Hkv, U = a.S * Hkv, G = a.G, T = a.T, R = G * T, Hq = Hkv * G;
  const int NC = gridDim.x, cta = blockIdx.x;
  const VLayout L = verify_layout(D, U, R);
  const int CK = L.ck, CV = L.cv, R8 = L.rb / 128;
  const uint32_t vring = sbase + L.ring_off + CK * kKChunk;
  int* PT = reinterpret_cast<int*>(smem + L.tab_off);   // [U + 1] tile prefix
  int* NK = PT + U + 1;                                   // [U] prefix keys per unit
  int* TROW = reinterpret_cast<int*>(smem + L.trow_off);  // [kTileRing][8] first tensor row of each group
  int* TMASK = TROW + kTileRing * 8;                      // [kTileRing][8] valid rows of each group
  int* VMASK = TMASK + kTileRing * 8;                     // the same, written by the V copy warp
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc_off + 16);
  const uint32_t bars = sbase + L.bar_off;

  // ---- unit table (caller metadata only)
  for (int u = threadIdx.x; u < U; u += kVThreads) {
    const int s = u / Hkv;
    int n;
    if (c.paged) {
      n = c.seq_len[s];
      const int cap = min(a.max_len, c.bt_stride * c.P);
      if (n < 0 || n > cap) {
        if (cta == 0 && u - s * Hkv == 0) raise_error(a.err, ERR_LENGTH);
        n = n < 0 ? 0 : cap;
      }
    } else {
      // a ring: every slot is scanned (the valid ones are masked in), none
      // when the ring is empty or its metadata is out of range
      const int cnt = c.ring_count[s], hd = c.ring_head[s];
      const int row = c.stream_rows ? c.stream_rows[s] : s;
      const bool bad = cnt < 0 || cnt > c.R || hd < 0 || hd >= c.R || row < 0 || row >= c.n_rows;
      if (bad && cta == 0 && u - s * Hkv == 0) raise_error(a.err, ERR_INDEX);
      n = (bad || cnt == 0) ? 0 : c.R;
    }
    NK[u] = n;
    PT[u + 1] = (n + KT - 1) / KT;
  }
  if (threadIdx.x == 0) {
    PT[0] = 0;
    *abort_flag = 0;
    for (int b = 0; b < kMaxK; ++b) {
      mbar_init(bars + 8 * (B_KFULL + b), 1);
      mbar_init(bars + 8 * (B_KFREE + b), 1);
    }
    for (int b = 0; b < kMaxV; ++b) {
      mbar_init(bars + 8 * (B_VFULL + b), 1);
      mbar_init(bars + 8 * (B_VCONV + b), kConvWarps);
      mbar_init(bars + 8 * (B_VFREE + b), 1);
    }
    mbar_init(bars + 8 * B_QLO, 1);
    mbar_init(bars + 8 * B_QHI, kSoftWarps);
    mbar_init(bars + 8 * B_QFREE, 1);
    mbar_init(bars + 8 * B_SFULL, 1);
    mbar_init(bars + 8 * B_SFREE, kSoftWarps);
    mbar_init(bars + 8 * B_PFULL, kSoftWarps);
    mbar_init(bars + 8 * B_PVDONE, 1);
    mbar_init(bars + 8 * B_OFREE, kSoftWarps);
    mbar_init(bars + 8 * B_FINAL, 2);  // one commit per issuing thread
    fence_mbar_init();
  }
  if (threadIdx.x == kTmaWarp * 32) {
    prefetch_tmap(&a.tmap_k);
    prefetch_tmap(&a.tmap_v);
    prefetch_tmap(&a.tmap_q);
  }
  __syncthreads();
  block_scan_inclusive<kVThreads>(PT + 1, U);
  const int Ttot = PT[U];
  // stream-K over the units' tiles, each unit weighted with the fixed cost of
  // one segment of it (its q rows come in, the pipeline refills, its partial
  // output leaves tensor memory)
  const Split sp{PT, U, kVerifySegmentCost, NC, Ttot + static_cast<int64_t>(kVerifySegmentCost) * U};
  const int g0 = sp.tile_at(sp.bound(cta));
  const int g1 = sp.tile_at(sp.bound(cta + 1));
  if (cta == 0) {
    // for the combine: the tile prefix, then per unit the first CTA of its
    // span, the span's length and the partial slot of its first segment
    for (int u = threadIdx.x; u <= U; u += kVThreads) a.tiles[u] = PT[u];
    for (int u = threadIdx.x; u < U; u += kVThreads) {
      int c_lo = 0, c_hi = -1, first_slot = 0;
      unit_segments(sp, PT[u], PT[u + 1], u, c_lo, c_hi, first_slot);
      a.tiles[U + 1 + u] = c_lo;
      a.tiles[2 * U + 1 + u] = c_hi - c_lo + 1;
      a.tiles[3 * U + 1 + u] = first_slot;
    }
  }
  const int nt = g1 - g0;
  if (nt > 0 && warp == kMmaWarp) tc::alloc(sbase + L.misc_off, Col::TOTAL > 256 ? 512 : 256);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L.misc_off);
  const Waiter W{bars, abort_flag, a.err};
  // the unit of CTA tile k (global tile g0 + k), from the unit of an earlier tile
  auto unit_at = [&](int k, int u) {
    while (PT[u + 1] <= g0 + k) ++u;
    return u;
  };
  const int u_first = nt > 0 ? unit_of(PT, U, g0) : 0;

  // lane gi < 8 of a copy warp: first tensor row and valid rows of group gi
  // of tile k of unit u (one page-table load)
  auto group_of = [&](int k, int u, int& row, int& mask) {
    row = mask = 0;
    if (lane >= 8 || k < 0 || k >= nt) return;
    const int s = u / Hkv, j = u - s * Hkv;
    const int t0 = ((g0 + k) - PT[u]) * KT + lane * 16;
    const int valid = min(16, NK[u] - t0);
    if (valid <= 0) return;
    if (!c.paged) {
      // slots t0 .. t0 + 15 of the ring; slot x is valid when it is one of
      // the `count` slots before `head`
      const int cnt = c.ring_count[s], hd = c.ring_head[s];
      const int rrow = c.stream_rows ? c.stream_rows[s] : s;
      uint32_t m = 0;
      for (int b = 0; b < valid; ++b) {
        const int age = ((t0 + b - hd + cnt) % c.R + c.R) % c.R;  // 0 = the oldest valid slot
        if (age < cnt) m |= 1u << b;
      }
      row = (rrow * Hkv + j) * c.R + t0;
      mask = static_cast<int>(m);
      return;
    }
    int pg = c.block_table[static_cast<int64_t>(s) * c.bt_stride + t0 / c.P];
    if (pg < 0 || pg >= c.n_rows) {
      raise_error(a.err, ERR_INDEX);
      pg = 0;
    }
    row = (pg * Hkv + j) * c.P + t0 % c.P;
    mask = static_cast<int>((1u << valid) - 1u);
  };
  if (nt > 0 && (warp == kTmaWarp || warp == kTmaVWarp)) {
    // ================= TMA: K (and each segment's q_lo rows) or V, one warp each =================
    // Each tile's group rows are worked out one tile ahead, so that no
    // page-table load waits on the issue path.
    const bool is_v = warp == kTmaVWarp;
    const int nring = is_v ? CV : CK;
    const int b_full = is_v ? B_VFULL : B_KFULL, b_free = is_v ? B_VFREE : B_KFREE;
    int* MASKS = is_v ? VMASK : TMASK;
    const uint64_t policy = l2_evict_first_policy();
    int u = u_first, seg = -1, issued = 0;
    int nrow, nmask;
    group_of(0, u, nrow, nmask);
    // The next tile's page-table loads are issued after this tile's copies,
    // so their latency falls inside the waits for free slots.
    bool waited = false, ok = true;
    for (int k = 0; k < nt && ok; ++k) {
      const int e = (k % kTileRing) * 8;
      const int un = unit_at(k, u);
      const bool new_seg = un != u || k == 0;
      u = un;
      int rows[8];
#pragma unroll
      for (int gi = 0; gi < 8; ++gi) rows[gi] = __shfl_sync(0xffffffffu, nrow, gi);
      if (lane < 8) MASKS[e + lane] = nmask;
      if (!is_v && lane < 8) TROW[e + lane] = nrow;
      __syncwarp();
      if (lane == 0) {
        // K(k): one slot per 64-dim region, one box per loaded group;
        // V(k): one slot per 16-key group, one box (all dims) when it has keys
        const int per_tile = is_v ? 8 : NREG;
        for (int ch = 0; ch < per_tile && ok; ++ch) {
          const int idx = k * per_tile + ch, slot = idx % nring;
          if (idx >= nring && !W.wait(b_free + slot, ((idx / nring) - 1) & 1)) {
            ok = false;
            break;
          }
          const uint32_t bar = bars + 8 * (b_full + slot);
          if (!is_v) {
            const uint32_t dst = sbase + L.ring_off + slot * kKChunk;
            int n = 0;
            for (int gi = 0; gi < 8; ++gi) n += MASKS[e + gi] != 0;
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n) * 2048u);
            for (int gi = 0; gi < 8; ++gi)
              if (MASKS[e + gi] != 0) tma_load_2d(dst + gi * 2048, &a.tmap_k, 64 * ch, rows[gi], bar, policy);
          } else {
            const bool any = MASKS[e + ch] != 0;
            mbar_arrive_expect_tx(bar, any ? static_cast<uint32_t>(VG) : 0u);
            if (any) tma_load_3d(vring + slot * VG, &a.tmap_v, 0, rows[ch], 0, bar, policy);
          }
          issued = idx + 1;
        }
        if (ok && new_seg && !is_v) {
          // the segment's q_lo rows once its previous segment's Q K^T
          // completed; the first ones once the prologue that writes them has
          if (!waited) {
            pdl_wait();
            waited = true;
          }
          ++seg;
          if (seg > 0 && !W.wait(B_QFREE, (seg - 1) & 1)) ok = false;
          if (ok) {
            const int s = u / Hkv, j = u - s * Hkv;
            const uint32_t bar = bars + 8 * B_QLO;
            mbar_arrive_expect_tx(bar, NREG * static_cast<uint32_t>(R) * 128u);
            for (int rr = 0; rr < NREG; ++rr)
              tma_load_4d(sbase + L.qlo_off + rr * L.rb, &a.tmap_q, 64 * rr, j * G, s * T, 1, bar, policy);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (k + 1 < nt) group_of(k + 1, unit_at(k + 1, u), nrow, nmask);
    }
    // Copies still in flight exist only when a role gave up: let the latest
    // copy into every slot and the last q copy land before the CTA exits.
    if (lane == 0 && *abort_flag) {
      for (int idx = max(0, issued - nring); idx < issued; ++idx)
        mbar_wait_bounded(bars + 8 * (b_full + idx % nring), (idx / nring) & 1);
      if (!is_v && seg >= 0) mbar_wait_bounded(bars + 8 * B_QLO, seg & 1);
    }
    __syncwarp();
  } else if (nt > 0 && warp >= kConv0 && warp < kConv0 + kConvWarps) {
    // ================= converters: each landed V chunk bf16 -> fp16 in place =================
    const int ct = threadIdx.x - kConv0 * 32;  // 0 .. 127
    uint32_t mag = 0;
    bool ok = true;
    for (int k = 0; k < nt && ok; ++k) {
      const int e = (k % kTileRing) * 8;
      for (int gi = 0; gi < 8; ++gi) {
        const int idx = k * 8 + gi, slot = idx % CV;
        if (!__all_sync(0xffffffffu, W.wait(B_VFULL + slot, (idx / CV) & 1))) {
          ok = false;
          break;
        }
        uint8_t* base = smem + L.ring_off + CK * kKChunk + slot * VG;
        const uint32_t vmask = static_cast<uint32_t>(VMASK[e + gi]);
#pragma unroll
        for (int i = 0; i < VG / 16 / 128; ++i) {
          // [region][16 rows][128 B]: rows outside the prefix become 0
          const int p = ct + i * 128;
          if ((vmask >> ((p >> 3) & 15)) & 1)
            convert16(base + p * 16, mag);
          else
            *reinterpret_cast<uint4*>(base + p * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (B_VCONV + slot));
      }
    }
    // fp16 holds bf16 values below 65504 in magnitude exactly (bf16 0x4780 = 65536)
    const bool ovf = (mag & 0xffffu) >= 0x4780u || (mag >> 16) >= 0x4780u;
    if (__any_sync(0xffffffffu, ovf) && lane == 0) raise_error(a.err, ERR_RANGE);
  } else if (nt > 0 && (warp == kMmaWarp || warp == kPvWarp)) {
    // ================= MMA issue: Q K^T from one thread, P V from another =================
    // The two chains run apart: Q K^T(k + 1) is issued as soon as K(k + 1)
    // has landed and the softmax warps hold S(k), whether or not P V(k) can
    // go yet (it waits for P(k) and V(k)); P V(k) waits for nothing of
    // K(k + 1). (In one issuing thread, P V(k) would sit behind Q K^T(k + 1)
    // and so behind K(k + 1)'s copies: 112.7 -> 108.5 us per tree-verify call.)
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::f16_idesc(VM, KT, 1, false);  // bf16; B = K: K-major
      constexpr uint32_t idesc_pv = tc::f16_idesc(VM, D, 0, true);    // B = V: D-contiguous
      int u = u_first, seg = -1;
      auto qk = [&](int k) -> bool {
        const int un = unit_at(k, u);
        const bool seg_first = un != u || k == 0;
        u = un;
        const bool seg_last = k == nt - 1 || g0 + k + 1 >= PT[u + 1];
        if (seg_first) {
          ++seg;
          if (!W.wait(B_QLO, seg & 1) || !W.wait(B_QHI, seg & 1)) return false;
        }
        // S is free once the softmax warps hold the previous tile's scores
        if (k > 0 && !W.wait(B_SFREE, (k - 1) & 1)) return false;
        for (int ch = 0; ch < NREG; ++ch) {
          const int idx = k * NREG + ch, slot = idx % CK;
          if (!W.wait(B_KFULL + slot, (idx / CK) & 1)) return false;  // K is used as it landed
          tc::fence_after();
          const uint32_t kc = sbase + L.ring_off + slot * kKChunk;
          const uint32_t qc = sbase + L.qlo_off + ch * L.rb;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t kdesc = tc::sw128_desc(kc + kk * 32, 16, 1024);
            tc::mma_ts(tmem + Col::S, tmem + Col::Q + (4 * ch + kk) * 8, kdesc, idesc_qk, ch > 0 || kk > 0);
            tc::mma(tmem + Col::S, tc::sw128_desc(qc + kk * 32, 16, 1024), kdesc, idesc_qk, true);
          }
          tc::commit(bars + 8 * (B_KFREE + slot));
        }
        tc::commit(bars + 8 * B_SFULL);
        if (seg_last) tc::commit(bars + 8 * B_QFREE);
        return true;
      };
      int pv_u = u_first, pv_seg = -1;
      auto pv = [&](int k) -> bool {
        const int un = unit_at(k, pv_u);
        const bool seg_first = un != pv_u || k == 0;
        pv_u = un;
        if (seg_first) ++pv_seg;
        if (!W.wait(B_PFULL, k & 1)) return false;
        if (seg_first && pv_seg > 0 && !W.wait(B_OFREE, (pv_seg - 1) & 1)) return false;
        for (int grp = 0; grp < 8; ++grp) {  // 16-key group of the tile
          const int idx = k * 8 + grp, slot = idx % CV;
          if (!W.wait(B_VCONV + slot, (idx / CV) & 1)) return false;
          tc::fence_after();
          const uint64_t pdesc = tc::sw128_desc(sbase + L.p_off + (grp >> 2) * L.rb + (grp & 3) * 32, 16, 1024);
          tc::mma(tmem + Col::O, pdesc, tc::sw128_desc(vring + slot * VG, 2048, 1024), idesc_pv,
                  !(seg_first && grp == 0));
          tc::commit(bars + 8 * (B_VFREE + slot));
        }
        tc::commit(bars + 8 * B_PVDONE);
        return true;
      };
      bool ok = true;
      if (warp == kMmaWarp) {
        for (int k = 0; k < nt && ok; ++k) ok = qk(k);
      } else {
        for (int k = 0; k < nt && ok; ++k) ok = pv(k);
      }
      // every MMA issued has completed before the tensor memory is freed
      tc::commit(bars + 8 * B_FINAL);
      if (!mbar_wait_bounded(bars + 8 * B_FINAL, 0)) raise_error(a.err, ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (nt > 0 && warp < kSoftWarps) {
    // ================= softmax: row t = 32 (w % 4) + lane, keys of half w / 4 =================
    const int q4 = warp & 3, kh = warp >> 2;
    const int t = 32 * q4 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    float* XMAX = reinterpret_cast<float*>(smem + L.xch_off);  // [2][2][128]
    float* XL = XMAX + 512;                                     // [2][128]
    // the two warps of a lane quarter (the two key halves of its rows) meet
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(1 + q4) : "memory"); };
    // unit u's q_hi rows into TMEM (the A operand of the first Q K^T MMA of
    // every 16 dims; rows past R are zero); each key half writes half the dims
    auto load_qhi = [&](int u) {
      const int s = u / Hkv, j = u - s * Hkv;
      const uint16_t* src = nullptr;
      if (t < R) {
        const int i = t / G, g = t - i * G;  // rows as the q_lo box lays them out: i * G + g
        src = a.qhl + ((static_cast<int64_t>(s) * T + i) * Hq + j * G + g) * D;
      }
#pragma unroll 1
      for (int c32 = kh * (D / 128); c32 < (kh + 1) * (D / 128); ++c32) {
        uint32_t qv[32];  // bf16 pairs, the lower dim in the low half
#pragma unroll
        for (int x = 0; x < 32; x += 4) {
          uint4 y = make_uint4(0u, 0u, 0u, 0u);
          if (src) y = *reinterpret_cast<const uint4*>(src + 64 * c32 + 2 * x);
          qv[x] = y.x;
          qv[x + 1] = y.y;
          qv[x + 2] = y.z;
          qv[x + 3] = y.w;
        }
        tc::st32(tmem + lane_off + Col::Q + 32 * c32, qv);
      }
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8 * B_QHI);
    };
    pdl_wait();  // q is written by the prologue
    load_qhi(u_first);
    int u = u_first, seg = -1;
    float m_ref = -INFINITY, l = 0.f;  // l: this half's share of the row sum
    // Ring layers: a row at depth d sees the newest min(count, R - d) entries,
    // what its path's d entries leave of the ring: `drop` of its oldest valid
    // slots (those at age < drop from `oldest`) are masked for this row.
    int drop = 0, oldest = 0;
    uint8_t* pbase = smem + L.p_off + kh * L.rb;  // P's key region of this half
    for (int k = 0; k < nt; ++k) {
      const int un = unit_at(k, u);
      const bool seg_first = un != u || k == 0;
      u = un;
      const bool seg_last = k == nt - 1 || g0 + k + 1 >= PT[u + 1];
      if (seg_first) {
        ++seg;
        m_ref = -INFINITY;
        l = 0.f;
        if (!c.paged && t < R) {
          const int s = u / Hkv, i = t / G;
          int depth = 0, node = i;
          for (int steps = 0; steps < T; ++steps) {
            const int p = a.parent[s * T + node];
            if (p < 0 || p >= node) break;  // (a bad parent is reported by the prologue)
            ++depth;
            node = p;
          }
          const int cnt = c.ring_count[s];
          drop = max(0, cnt - c.R + depth);
          oldest = ((c.ring_head[s] - cnt) % c.R + c.R) % c.R;
        }
      }
      if (!__all_sync(0xffffffffu, W.wait(B_SFULL, k & 1))) break;
      tc::fence_after();
      // this row's scores of the half-tile, then S is free for the next Q K^T
      float sv[64];
      tc::ld64(tmem + lane_off + Col::S + 64 * kh, *reinterpret_cast<uint32_t(*)[64]>(sv));
      tc::wait_ld();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8 * B_SFREE);
      // the next unit's q_hi, as soon as this segment's Q K^T completed
      // (already true: it completed before this tile's scores were read)
      if (seg_last && k + 1 < nt) {
        if (!__all_sync(0xffffffffu, W.wait(B_QFREE, seg & 1))) break;
        load_qhi(unit_at(k + 1, u));
      }
      // (the tile's group masks were written before its first copy was issued)
      const int e = (k % kTileRing) * 8 + 4 * kh;
      const uint32_t km0 = t < R ? static_cast<uint32_t>(TMASK[e]) | (static_cast<uint32_t>(TMASK[e + 1]) << 16) : 0u;
      const uint32_t km1 = t < R ? static_cast<uint32_t>(TMASK[e + 2]) | (static_cast<uint32_t>(TMASK[e + 3]) << 16) : 0u;
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (drop > 0) {
        // the masked slots are [oldest, oldest + drop) cyclically: as sv
        // indices [lo, hi), and [0, hi2) for the part that wraps to slot 0
        const int key0 = ((g0 + k) - PT[u]) * KT + 64 * kh;  // ring slot of sv[0]
        const int lo = oldest - key0, hi = lo + drop, hi2 = hi - c.R;
#pragma unroll
        for (int x = 0; x < 64; ++x)
          if ((x >= lo && x < hi) || x < hi2) sv[x] = -INFINITY;
      }
#pragma unroll
      for (int x = 0; x < 64; ++x) {
        if (!(((x < 32 ? km0 : km1) >> (x & 31)) & 1u)) sv[x] = -INFINITY;
        mx[x & 3] = fmaxf(mx[x & 3], sv[x]);
      }
      // (two buffers by tile parity: a half may start the next tile while its
      // partner still reads this one's)
      float* xm = XMAX + (k & 1) * 256;
      xm[kh * 128 + t] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      pair_sync();
      const float tmax = fmaxf(xm[t], xm[128 + t]);
      const bool need = tmax > m_ref + kRescaleLog2;
      const float f = need ? exp2_fast(m_ref - tmax) : 1.f;  // 0 when the reference was -inf
      if (need) {
        l *= f;
        m_ref = tmax;
      }
      // P and O are free, and O complete, once the previous tile's P V completed
      if (k > 0 && !__all_sync(0xffffffffu, W.wait(B_PVDONE, (k - 1) & 1))) break;
      tc::fence_after();
      // Rows whose reference moved rescale their output so far (this half of
      // its columns). The TMEM loads and stores are warp-wide, so the warp
      // takes them together (factor 1 for the other rows).
      if (!seg_first && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int cc = kh * (D / 64); cc < (kh + 1) * (D / 64); ++cc) {
          uint32_t o[32];
          tc::ld32(tmem + lane_off + Col::O + cc * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * f);
          tc::st32(tmem + lane_off + Col::O + cc * 32, o);
        }
        tc::wait_st();
      }
      // probabilities in fp16 into P (row t, this half's 64 keys: one 128-byte
      // row, 16-byte chunks of 8 keys swizzled by the row); the row sum uses
      // the same rounded values
      float ls[2] = {0.f, 0.f};
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        uint32_t w4[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const float s0 = sv[8 * c8 + 2 * x], s1 = sv[8 * c8 + 2 * x + 1];
          const float p0 = s0 == -INFINITY ? 0.f : exp2_fast(s0 - m_ref);
          const float p1 = s1 == -INFINITY ? 0.f : exp2_fast(s1 - m_ref);
          const __half2 hp = __floats2half2_rn(p0, p1);
          ls[x & 1] += __low2float(hp) + __high2float(hp);
          w4[x] = *reinterpret_cast<const uint32_t*>(&hp);
        }
        if (t < R8)  // (the region holds R8 rows)
          *reinterpret_cast<uint4*>(pbase + t * 128 + ((c8 ^ (t & 7)) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      l += ls[0] + ls[1];
      fence_proxy_async_smem();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8 * B_PFULL);
      if (seg_last) {
        // ---- the segment's partial state: o (relative to the reference), m, l
        if (!__all_sync(0xffffffffu, W.wait(B_PVDONE, k & 1))) break;
        tc::fence_after();
        const int slot = seg == 0 ? cta : NC + u;
        float* dst = nullptr;
        if (t < R) {
          const int i = t / G, g = t - i * G;
          dst = a.part + (static_cast<int64_t>(slot) * R + g * T + i) * row_stride<D>();
        }
#pragma unroll 1
        for (int cc = kh * (D / 64); cc < (kh + 1) * (D / 64); ++cc) {
          uint32_t o[32];
          tc::ld32(tmem + lane_off + Col::O + cc * 32, o);
          tc::wait_ld();
          if (dst) {
#pragma unroll
            for (int x = 0; x < 32; x += 4)
              *reinterpret_cast<float4*>(dst + cc * 32 + x) =
                  make_float4(__uint_as_float(o[x]), __uint_as_float(o[x + 1]), __uint_as_float(o[x + 2]),
                              __uint_as_float(o[x + 3]));
          }
        }
        XL[kh * 128 + t] = l;
        pair_sync();
        if (dst && kh == 0) {
          dst[D] = m_ref;
          dst[D + 1] = XL[t] + XL[128 + t];
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * B_OFREE);
      }
    }
  }

  tc::fence_before();
  __syncthreads();
  if (nt > 0 && warp == kMmaWarp) {
    tc::fence_after();
    tc::dealloc(tmem, Col::TOTAL > 256 ? 512 : 256);
  }
  // The combine may begin once every CTA of this pass has triggered, and each
  // one does so only after the prologue has completed: so the combine reads
  // the rotated q and window keys before waiting for this pass.
  pdl_wait();
  pdl_trigger();
}

// ---------------------------------------------------------------- combine

template <int D>
__global__ void __launch_bounds__(256, 6) verify_combine_kernel(const VerifyCombineArgs a) {
  constexpr int EPL = D / 32;  // dims per lane
  __shared__ int par_s[16];
  __shared__ int path_s[16];
  __shared__ int npath_s;
  const int i = blockIdx.x, j = blockIdx.y, s = blockIdx.z;
  const int g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.G, T = a.T, Hkv = a.Hkv, Hq = Hkv * G, R = G * T, h = j * G + g;
  const int64_t tok = static_cast<int64_t>(s) * T + i;          // row of the workspace arrays
  const int64_t ctok = static_cast<int64_t>(s) * a.in_T + a.row0 + i;  // row of the caller's v, gate, out
  // (a prefill chunk's rows past the stream's new tokens are neither read nor stored)
  const bool stored = a.rows_valid ? i < a.rows_valid[s] : true;
  const CacheView& c = a.c;

  // ---- caller inputs: tree, gate, prefix length, write-back target
  if (threadIdx.x < T) par_s[threadIdx.x] = a.parent[static_cast<int64_t>(s) * T + threadIdx.x];
  __syncthreads();
  if (threadIdx.x == 0) {
    int np = 0, node = i;
    path_s[np++] = node;
    for (int steps = 0; steps < T; ++steps) {
      const int p = par_s[node];
      if (p < 0) break;
      if (p >= node) {
        raise_error(a.err, ERR_INDEX);
        break;
      }
      node = p;
      path_s[np++] = node;
    }
    npath_s = np;
  }
  float sig = 1.f;
  if (a.gate && stored) sig = 1.f / (1.f + expf(-bf16_to_f32(a.gate[ctok * Hq + h])));
  int64_t wb_off = -1;
  if (a.write_back && c.paged && g == 0) {  // (ring layers commit the accepted path instead)
    int n = c.seq_len[s];
    const int cap = min(a.max_len, c.bt_stride * c.P);
    n = n < 0 ? 0 : (n > cap ? cap : n);
    const int idx = n + i;
    const int pi = idx / c.P;
    const int pg = pi < c.bt_stride ? c.block_table[static_cast<int64_t>(s) * c.bt_stride + pi] : -1;
    if (pg >= 0 && pg < c.n_rows)
      wb_off = ((static_cast<int64_t>(pg) * Hkv + j) * c.P + idx % c.P) * D;
    else if (lane == 0)
      raise_error(a.err, ERR_INDEX);
  }
  __syncthreads();
  const int np = npath_s;

  // ---- before waiting for the prefix pass (the prologue it waited for has
  // completed): the row's tree path - itself and its ancestors - scored in
  // fp32 and joined as a softmax state (M, L, acc) of its own
  float q[EPL];
  {
    const float* src = a.qhat + (tok * Hq + h) * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; e += 4) {
      const float4 x = *reinterpret_cast<const float4*>(src + e);
      q[e] = x.x; q[e + 1] = x.y; q[e + 2] = x.z; q[e + 3] = x.w;
    }
  }
  // path nodes four at a time: their rows' loads go out together (the
  // scores stay in registers: every index below is a compile-time one)
  constexpr int kPathBatch = 4;
  float sw[16];
  float M = -INFINITY;
#pragma unroll
  for (int p0 = 0; p0 < 16; p0 += kPathBatch) {
    if (p0 >= np) break;
    uint32_t kw[kPathBatch][EPL / 2];
#pragma unroll
    for (int b = 0; b < kPathBatch; ++b) {
      if (p0 + b >= np) break;
      const uint16_t* kp = a.khat + ((static_cast<int64_t>(s) * T + path_s[p0 + b]) * Hkv + j) * D + lane * EPL;
#pragma unroll
      for (int e = 0; e < EPL; e += 2) kw[b][e / 2] = *reinterpret_cast<const uint32_t*>(kp + e);
    }
#pragma unroll
    for (int b = 0; b < kPathBatch; ++b) {
      if (p0 + b >= np) break;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; e += 2) {
        dot = fmaf(q[e], bf16_lo(kw[b][e / 2]), dot);
        dot = fmaf(q[e + 1], bf16_hi(kw[b][e / 2]), dot);
      }
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, w);
      sw[p0 + b] = dot;
      M = fmaxf(M, dot);
    }
  }
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float L = 0.f;  // relative to M
#pragma unroll
  for (int p0 = 0; p0 < 16; p0 += kPathBatch) {
    if (p0 >= np) break;
    uint32_t vw[kPathBatch][EPL / 2];
#pragma unroll
    for (int b = 0; b < kPathBatch; ++b) {
      if (p0 + b >= np || !stored) break;  // (a stored row's ancestors lie within the caller's rows)
      const uint16_t* vp =
          a.v + ((static_cast<int64_t>(s) * a.in_T + a.row0 + path_s[p0 + b]) * Hkv + j) * D + lane * EPL;
#pragma unroll
      for (int e = 0; e < EPL; e += 2) vw[b][e / 2] = *reinterpret_cast<const uint32_t*>(vp + e);
    }
#pragma unroll
    for (int b = 0; b < kPathBatch; ++b) {
      if (p0 + b >= np) break;
      const float w = exp2_fast(sw[p0 + b] - M);
      L += w;
      if (!stored) continue;
#pragma unroll
      for (int e = 0; e < EPL; e += 2) {
        acc[e] = fmaf(w, bf16_lo(vw[b][e / 2]), acc[e]);
        acc[e + 1] = fmaf(w, bf16_hi(vw[b][e / 2]), acc[e + 1]);
      }
    }
  }

  pdl_wait();  // the prefix partials and their layout
  pdl_trigger();

  // ---- the prefix segments of this unit (row r = g * T + i), merged online
  const int U = a.S * Hkv, u = s * Hkv + j, NC = a.split_ctas;
  const int Ttot = a.tiles[U];
  const int c_lo = a.tiles[U + 1 + u], S = a.tiles[2 * U + 1 + u], first_slot = a.tiles[3 * U + 1 + u];
  const int64_t W = Ttot + static_cast<int64_t>(kVerifySegmentCost) * U;  // the split's weighted length
  const int r = g * T + i;
  auto seg_row = [&](int k) -> const float* {
    const int slot = k == 0 ? first_slot : c_lo + k;
    return a.part + (static_cast<int64_t>(slot) * R + r) * row_stride<D>();
  };
  auto seg_ok = [&](int k) -> bool {  // a CTA strictly inside the span holds tiles iff its range is not empty
    if (k >= S) return false;
    if (k == 0) return true;
    const int64_t cc = c_lo + k;
    return cc * W / NC < (cc + 1) * W / NC;
  };
  constexpr int SB = 2;  // segments whose loads go out together
  for (int k0 = 0; k0 < S; k0 += SB) {
    float mk[SB], lk[SB], ok[SB][EPL];
#pragma unroll
    for (int b = 0; b < SB; ++b) {
      mk[b] = -INFINITY;
      lk[b] = 0.f;
      if (seg_ok(k0 + b)) {
        const float* pr = seg_row(k0 + b);
        mk[b] = __ldcg(pr + D);
        lk[b] = __ldcg(pr + D + 1);
#pragma unroll
        for (int e = 0; e < EPL; e += 4) {
          const float4 x = __ldcg(reinterpret_cast<const float4*>(pr + lane * EPL + e));
          ok[b][e] = x.x; ok[b][e + 1] = x.y; ok[b][e + 2] = x.z; ok[b][e + 3] = x.w;
        }
      }
    }
    float Mn = M;
#pragma unroll
    for (int b = 0; b < SB; ++b) Mn = fmaxf(Mn, mk[b]);
    const float f = exp2_fast(M - Mn);  // M is finite: the row's own score is in it
    L *= f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] *= f;
#pragma unroll
    for (int b = 0; b < SB; ++b) {
      if (mk[b] == -INFINITY) continue;
      const float w = exp2_fast(mk[b] - Mn);
      L = fmaf(w, lk[b], L);
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w, ok[b][e], acc[e]);
    }
    M = Mn;
  }
  const float scale = sig / L;
  float* dst = a.out + (ctok * Hq + h) * D + lane * EPL;
  if (stored) {
#pragma unroll
    for (int e = 0; e < EPL; e += 4)
      *reinterpret_cast<float4*>(dst + e) =
          make_float4(acc[e] * scale, acc[e + 1] * scale, acc[e + 2] * scale, acc[e + 3] * scale);
  }

  // ---- write-back of this node's entry at token index prefix_len + i
  if (wb_off >= 0) {
    const uint16_t* kh = a.khat + (tok * Hkv + j) * D + lane * EPL;
    const uint16_t* vv = a.v + (ctok * Hkv + j) * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; e += 4) {
      *reinterpret_cast<uint2*>(c.k + wb_off + lane * EPL + e) = *reinterpret_cast<const uint2*>(kh + e);
      *reinterpret_cast<uint2*>(c.v + wb_off + lane * EPL + e) = *reinterpret_cast<const uint2*>(vv + e);
    }
  }
}

template <int D>
cudaError_t verify_split_launch(const VerifySplitArgs& a, cudaStream_t s) {
  static std::atomic<uint64_t> opted{0};
  const cudaError_t e = opt_in_smem(verify_split_kernel<D>, kSmemLimit, opted);
  if (e != cudaSuccess) return e;
  const VLayout L = verify_layout(D, a.S * a.Hkv, a.G * a.T);
  if (L.cv < 4 || L.total > kSmemLimit) return cudaErrorNotSupported;
  return launch_pdl(verify_split_kernel<D>, dim3(a.ctas), dim3(kVThreads), static_cast<size_t>(L.total), s, a);
}

}  // namespace

cudaError_t launch_verify_split(const VerifySplitArgs& a, int D, cudaStream_t s) {
  if (a.G * a.T > VM || a.T > 16 || a.S * a.Hkv > kVerifyMaxUnits) return cudaErrorNotSupported;
  if (D == 256) return verify_split_launch<256>(a, s);
  if (D == 128) return verify_split_launch<128>(a, s);
  return cudaErrorNotSupported;
}

cudaError_t launch_verify_combine(const VerifyCombineArgs& a, int D, cudaStream_t s) {
  if (a.G > 8 || a.T > 16) return cudaErrorNotSupported;
  dim3 grid(a.T, a.Hkv, a.S);
  dim3 block(32 * a.G);
  if (D == 256) return launch_pdl(verify_combine_kernel<256>, grid, block, 0, s, a);
  if (D == 128) return launch_pdl(verify_combine_kernel<128>, grid, block, 0, s, a);
  return cudaErrorNotSupported;
}

}  // namespace dattn
