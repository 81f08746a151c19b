// Tree verify: S streams x T draft rows, each row under its own tree mask
// ("TensorFold PR #608": verify rounds take every stream's window together, up
// to 16 streams of 16 rows). Row i of stream s sits at position
// prefix_len + depth(i) and attends to the stream's whole paged prefix, its
// ancestors in the tree and itself.
//
// Two passes after the RoPE prologue:
//  * verify_split_kernel - the prefix, on the 5th-generation tensor cores. The
//    G*T query rows of one (stream, KV head) unit share every prefix key, so a
//    unit is one 128-row MMA tile (G*T <= 128): S = Q K^T into tensor memory
//    (TMEM), an online softmax by four warps (thread t owns row t), then
//    O += P V accumulated in TMEM. Work is split stream-K over all units'
//    32-key tiles (one CTA per SM).
//    Operands are fp16: a TMA warp brings the bf16 K/V rows of each 16-key
//    group (contiguous within a page) by one bulk copy each into one of three
//    row-major bf16 stages, and eight producer warps convert each tile into
//    one of three fp16 operand buffers in the 128-byte-swizzled layout the
//    MMAs read (exact for |x| < 65504).
//    A stage is refilled as soon as it is converted, so the copies in flight
//    do not wait for the tile's MMAs; an operand buffer is held from its
//    conversion until its PV completes. q and P are rounded to fp16. (fp16 keeps the
//    error of q and P rounding under the tolerance at every prefix length;
//    bf16 operands do not at short prefixes.) The accumulator is rescaled
//    lazily: only when a row's maximum grows by more than 2^8.
//  * verify_combine_kernel - per (stream, row, KV head): merges the prefix
//    segments, scores the row's tree path in fp32 and joins it in score
//    space, applies the gate, stores fp32 and writes the window entries back.
#include <cuda_fp16.h>

#include "common.cuh"
#include "mma.cuh"
#include "tc.cuh"

namespace dattn {

namespace {

constexpr int VM = 128;              // MMA rows (G*T <= VM)
constexpr int VNK = kVerifyTileKeys; // keys per tile
constexpr int NST = 3;               // bf16 K/V stages the TMA fills (released once converted)
constexpr int NWB = 3;               // fp16 operand buffers (released once their PV completes)
constexpr int NSB = 4;               // score buffers in tensor memory (each later holds its tile's P)
constexpr int kWin = 32;             // tiles whose page rows the TMA warp resolves at once
constexpr int kSoftWarps = 4;        // softmax warps: TMEM lane quarters 0..3
constexpr int kProdWarps = 8;        // producer warps
constexpr int kMmaWarp = kSoftWarps + kProdWarps;
constexpr int kTmaWarp = kMmaWarp + 1;   // issues the prefix tiles' TMA copies
constexpr int kPvWarp = kTmaWarp + 1;    // issues the P V MMAs (kMmaWarp issues Q K^T)
constexpr int kVThreads = (kPvWarp + 1) * 32;
constexpr float kRescaleLog2 = 8.f;  // lazy rescale threshold

// barrier indices
// (B_LOAD, B_EMPTY: one per bf16 stage; B_FULL, B_WFREE: one per fp16 operand
// buffer; B_SFULL, B_PFULL, B_SDONE: one per score buffer (its scores are in,
// its P is in, its PV has completed); B_PVDONE: PV(k) completed, by k & 1; one per
// probability buffer)
enum {
  B_LOAD = 0,
  B_EMPTY = B_LOAD + NST,
  B_FULL = B_EMPTY + NST,
  B_WFREE = B_FULL + NWB,
  B_SFULL = B_WFREE + NWB,
  B_PFULL = B_SFULL + NSB,
  B_SDONE = B_PFULL + NSB,
  B_PVDONE = B_SDONE + NSB,
  B_QREADY = B_PVDONE + 2,
  B_OFREE = B_QREADY + 1,
  B_COUNT = B_OFREE + 1
};

// A partial row is o[D], m, l, padded to a 16-byte multiple: D + 4 floats.
template <int D>
constexpr int row_stride() { return D + 4; }

template <int D>
struct VGeo {
  static constexpr int NREG = D / 64;                 // 64-dim (128-byte) regions per row
  static constexpr int KT_REG = VNK * 128;            // bytes of one K (or V) region
  static constexpr int KT_BYTES = NREG * KT_REG;
  static constexpr int ST_OFF = 0;                    // NST bf16 stages as the TMA wrote them
  static constexpr int ST_BYTES = 2 * KT_BYTES;       // K then V
  static constexpr int WB_OFF = ST_OFF + NST * ST_BYTES;  // NWB fp16 operand buffers, same layout
  static constexpr int BAR_OFF = WB_OFF + NWB * ST_BYTES;
  static constexpr int NBAR = B_COUNT;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8; // tmem slot, abort flag
  static constexpr int TAB_OFF = MISC_OFF + 16;
  static constexpr int SMEM = TAB_OFF + (2 * kVerifyMaxUnits + 1) * 4 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  // NSB score buffers of VNK columns; P of a tile is written over its scores
  // once they are read (the buffer's first VNK/2 columns, the A operand of P V)
  static constexpr uint32_t S_COL = 0;
  static constexpr uint32_t S_BUF = VNK;              // columns per score buffer
  static constexpr uint32_t Q_COL = NSB * S_BUF;      // q rows as the MMA's A: D/2 columns of fp16 pairs
  static constexpr uint32_t O_COL = 256;              // D columns of output
  static_assert(D == 128 || D == 256, "head_dim");
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
      if (global_timer_ns() - t0 > 2000000000ull) {
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


template <int D>
__global__ void __launch_bounds__(kVThreads, 1) verify_split_kernel(const __grid_constant__ VerifySplitArgs a) {
  using V = VGeo<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const CacheView& c = a.c;
  const int Hkv = a.Hkv, U = a.S * Hkv, G = a.G, T = a.T, R = G * T, Hq = Hkv * G;
  const int NC = gridDim.x, cta = blockIdx.x;
  int* Pt = reinterpret_cast<int*>(smem + V::TAB_OFF);  // [U + 1] tile prefix
  int* Nn = Pt + U + 1;                                   // [U] prefix keys per unit
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + V::MISC_OFF + 4);

  // ---- unit table (caller metadata only)
  for (int u = threadIdx.x; u < U; u += kVThreads) {
    const int s = u / Hkv;
    int n = c.seq_len[s];
    const int cap = min(a.max_len, c.bt_stride * c.P);
    if (n < 0 || n > cap) {
      if (cta == 0 && u - s * Hkv == 0) raise_error(a.err, ERR_LENGTH);
      n = n < 0 ? 0 : cap;
    }
    Nn[u] = n;
    Pt[u + 1] = (n + VNK - 1) / VNK;
  }
  if (threadIdx.x == 0) {
    Pt[0] = 0;
    *abort_flag = 0;
    for (int b = 0; b < NST; ++b) {
      mbar_init(sbase + V::BAR_OFF + 8 * (B_LOAD + b), 1);
      mbar_init(sbase + V::BAR_OFF + 8 * (B_EMPTY + b), kProdWarps);
    }
    for (int b = 0; b < NWB; ++b) {
      mbar_init(sbase + V::BAR_OFF + 8 * (B_FULL + b), kProdWarps);
      mbar_init(sbase + V::BAR_OFF + 8 * (B_WFREE + b), 1);
    }
    for (int b = 0; b < NSB; ++b) {
      mbar_init(sbase + V::BAR_OFF + 8 * (B_SFULL + b), 1);
      mbar_init(sbase + V::BAR_OFF + 8 * (B_PFULL + b), kSoftWarps);
      mbar_init(sbase + V::BAR_OFF + 8 * (B_SDONE + b), 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(sbase + V::BAR_OFF + 8 * (B_PVDONE + b), 1);
    mbar_init(sbase + V::BAR_OFF + 8 * B_QREADY, kSoftWarps);
    mbar_init(sbase + V::BAR_OFF + 8 * B_OFREE, kSoftWarps);
    fence_mbar_init();
  }
  __syncthreads();
  block_scan_inclusive<kVThreads>(Pt + 1, U);
  const int Ttot = Pt[U];
  // stream-K over the units' tiles, each unit weighted with the fixed cost of
  // one segment of it (at a segment end the whole tile pipeline drains, the
  // partial output leaves tensor memory and the next unit's q comes in)
  const Split sp{Pt, U, kVerifySegmentCost, NC, Ttot + static_cast<int64_t>(kVerifySegmentCost) * U};
  const int g0 = sp.tile_at(sp.bound(cta));
  const int g1 = sp.tile_at(sp.bound(cta + 1));
  if (cta == 0) {
    // for the combine: the tile prefix, then per unit the first CTA of its
    // span, the span's length and the partial slot of its first segment
    for (int u = threadIdx.x; u <= U; u += kVThreads) a.tiles[u] = Pt[u];
    for (int u = threadIdx.x; u < U; u += kVThreads) {
      int c_lo = 0, c_hi = -1, first_slot = 0;
      unit_segments(sp, Pt[u], Pt[u + 1], u, c_lo, c_hi, first_slot);
      a.tiles[U + 1 + u] = c_lo;
      a.tiles[2 * U + 1 + u] = c_hi - c_lo + 1;
      a.tiles[3 * U + 1 + u] = first_slot;
    }
  }
  if (warp == kMmaWarp) tc::alloc(sbase + V::MISC_OFF, V::TMEM_COLS);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + V::MISC_OFF);

  const int ntiles = g1 - g0;
  const Waiter W{sbase + V::BAR_OFF, abort_flag, a.err};

  if (ntiles > 0 && warp == kTmaWarp) {
    // ================= TMA: bf16 K/V page rows into the stage =================
    // Each 16-key group of a tile is 16 consecutive rows of one page (its size
    // is a multiple of 16): one contiguous bulk copy each for K and V, stored
    // row-major; the producers lay them out for the MMAs. Groups past the
    // prefix are not loaded; the producers zero their rows.
    // Lane x % 32 reads the page ids of tile x one 32-tile window ahead, so
    // that no page-table load sits between two tiles' copies; lane 0 issues.
    constexpr int NG = VNK / 16;
    const uint64_t policy = l2_evict_first_policy();
    auto fetch = [&](int x, int (&pg)[NG], int (&off)[NG]) -> int {  // returns the group count
#pragma unroll
      for (int gr = 0; gr < NG; ++gr) pg[gr] = off[gr] = 0;
      if (x >= ntiles) return 0;
      const int g = g0 + x;
      const int u = unit_of(Pt, U, g);
      const int s = u / Hkv, j = u - s * Hkv;
      const int k0 = (g - Pt[u]) * VNK;
      const int ng = (min(VNK, Nn[u] - k0) + 15) / 16;
      const int32_t* bt = c.block_table + static_cast<int64_t>(s) * c.bt_stride;
#pragma unroll
      for (int gr = 0; gr < NG; ++gr) {
        if (gr < ng) {
          const int t = k0 + gr * 16;
          const int pi = t / c.P;
          pg[gr] = bt[pi];  // used a window later: the load is not waited for here
          off[gr] = j * c.P + (t - pi * c.P);
        }
      }
      return ng;
    };
    int pg_c[NG], off_c[NG], pg_n[NG], off_n[NG];
    int ng_c = fetch(lane, pg_c, off_c);
    int ng_n = fetch(kWin + lane, pg_n, off_n);
    for (int k = 0; k < ntiles; ++k) {
      if (k > 0 && (k & (kWin - 1)) == 0) {
#pragma unroll
        for (int gr = 0; gr < NG; ++gr) {
          pg_c[gr] = pg_n[gr];
          off_c[gr] = off_n[gr];
        }
        ng_c = ng_n;
        ng_n = fetch(k + kWin + lane, pg_n, off_n);
      }
      const int st = k % NST;
      if (k >= NST && !__all_sync(0xffffffffu, W.wait(B_EMPTY + st, (k / NST - 1) & 1))) break;
      const int src = k & (kWin - 1);
      const int ngroups = __shfl_sync(0xffffffffu, ng_c, src);
      int rows[NG];
#pragma unroll
      for (int gr = 0; gr < NG; ++gr) {
        int pg = __shfl_sync(0xffffffffu, pg_c[gr], src);
        const int off = __shfl_sync(0xffffffffu, off_c[gr], src);
        if (gr < ngroups && (pg < 0 || pg >= c.n_rows)) {
          if (lane == 0) raise_error(a.err, ERR_INDEX);
          pg = 0;
        }
        rows[gr] = pg * Hkv * c.P + off;
      }
      if (lane == 0) {
        // one bulk copy per 16-key group of K and of V: 16 consecutive rows of
        // a page (8 KB at D = 256), row-major into the stage
        const uint32_t bar = sbase + V::BAR_OFF + 8 * (B_LOAD + st);
        const uint32_t stage = sbase + V::ST_OFF + st * V::ST_BYTES;
        constexpr uint32_t GB = 16u * D * 2u;  // bytes of one group
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(ngroups) * 2u * GB);
#pragma unroll
        for (int gr = 0; gr < NG; ++gr) {
          if (gr < ngroups) {
            const int64_t e0 = static_cast<int64_t>(rows[gr]) * D;
            bulk_copy_g2s(stage + gr * GB, c.k + e0, GB, bar, policy);
            bulk_copy_g2s(stage + V::KT_BYTES + gr * GB, c.v + e0, GB, bar, policy);
          }
        }
      }
      __syncwarp();
    }
  } else if (ntiles > 0 && warp >= kSoftWarps && warp < kMmaWarp) {
    // ================= producers: a staged bf16 tile -> fp16 operand buffer k % NWB =================
    // (row-major bf16 in, the MMAs' 128-byte-swizzled fp16 layout out)
    // The stage goes back to the TMA as soon as it is read; the operand buffer
    // is free again once the PV NWB tiles back has completed.
    const int pt = threadIdx.x - kSoftWarps * 32;         // 0 .. 255
    constexpr int CPR = D / 8;                            // 16-byte chunks per row
    constexpr int NCH = 2 * VNK * CPR;                    // chunks of a stage (K and V)
    constexpr int PER = NCH / (kProdWarps * 32);          // chunks per thread
    static_assert(NCH % (kProdWarps * 32) == 0, "whole chunks per thread");
    // this thread's chunks (the same positions in every tile): byte offset in
    // the row-major stage, in the swizzled operand buffer, and key row
    int soff[PER], coff[PER], crow[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = pt + i * kProdWarps * 32;
      const int which = e / (VNK * CPR);
      const int rem = e - which * (VNK * CPR);
      const int r = rem / CPR, ch = rem - r * CPR;
      soff[i] = which * V::KT_BYTES + r * (D * 2) + ch * 16;
      coff[i] = which * V::KT_BYTES + (ch >> 3) * V::KT_REG + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
      crow[i] = r;
    }
    uint32_t mag = 0;  // largest |x| seen, per 16-bit half (bf16 bit patterns)
    int u = unit_of(Pt, U, g0);
    for (int k = 0; k < ntiles; ++k) {
      const int st = k % NST, wb = k % NWB;
      if (!__all_sync(0xffffffffu, W.wait(B_LOAD + st, (k / NST) & 1))) break;
      if (k >= NWB && !__all_sync(0xffffffffu, W.wait(B_WFREE + wb, (k / NWB - 1) & 1))) break;
      const int g = g0 + k;
      while (Pt[u + 1] <= g) ++u;
      const int nvalid = min(VNK, Nn[u] - (g - Pt[u]) * VNK);
      const uint8_t* stage = smem + V::ST_OFF + st * V::ST_BYTES;
      uint8_t* obuf = smem + V::WB_OFF + wb * V::ST_BYTES;
      // all loads first, then the conversions and stores (rows past the prefix become zeros)
      uint4 w[PER];
#pragma unroll
      for (int i = 0; i < PER; ++i)
        w[i] = crow[i] < nvalid ? *reinterpret_cast<const uint4*>(stage + soff[i]) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        mag = __vmaxu2(mag, w[i].x & 0x7fff7fffu);
        mag = __vmaxu2(mag, w[i].y & 0x7fff7fffu);
        mag = __vmaxu2(mag, w[i].z & 0x7fff7fffu);
        mag = __vmaxu2(mag, w[i].w & 0x7fff7fffu);
        const uint4 h = make_uint4(cvt_pair_f16(bf16_lo(w[i].x), bf16_hi(w[i].x)),
                                   cvt_pair_f16(bf16_lo(w[i].y), bf16_hi(w[i].y)),
                                   cvt_pair_f16(bf16_lo(w[i].z), bf16_hi(w[i].z)),
                                   cvt_pair_f16(bf16_lo(w[i].w), bf16_hi(w[i].w)));
        *reinterpret_cast<uint4*>(obuf + coff[i]) = h;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(sbase + V::BAR_OFF + 8 * (B_FULL + wb));
        mbar_arrive(sbase + V::BAR_OFF + 8 * (B_EMPTY + st));
      }
    }
    // fp16 holds bf16 values below 65504 in magnitude exactly (bf16 0x4780 = 65536)
    const bool ovf = (mag & 0xffffu) >= 0x4780u || (mag >> 16) >= 0x4780u;
    if (__any_sync(0xffffffffu, ovf) && lane == 0) raise_error(a.err, ERR_RANGE);
  } else if (ntiles > 0 && warp == kMmaWarp) {
    // ================= Q K^T issue (one thread) =================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::f16_idesc(VM, VNK, 0, false);
      int u = unit_of(Pt, U, g0), prev_u = -1, seg = 0;
      for (int k = 0; k < ntiles; ++k) {
        const int g = g0 + k;
        while (Pt[u + 1] <= g) ++u;
        if (u != prev_u) {  // this unit's q rows are in place
          if (!W.wait(B_QREADY, seg & 1)) break;
          ++seg;
          prev_u = u;
        }
        const int sb = k % NSB, wb = k % NWB;
        if (!W.wait(B_FULL + wb, (k / NWB) & 1)) break;
        // the score buffer (and the P in it) is free once the PV NSB tiles back has completed
        if (k >= NSB && !W.wait(B_SDONE + sb, (k / NSB - 1) & 1)) break;
        tc::fence_after();
        const uint32_t kbase = sbase + V::WB_OFF + wb * V::ST_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t db = tc::sw128_desc(kbase + (kk >> 2) * V::KT_REG + (kk & 3) * 32, 16, 1024);
          tc::mma_ts(tmem + V::S_COL + sb * V::S_BUF, tmem + V::Q_COL + kk * 8, db, idesc_qk, kk > 0);
        }
        tc::commit(sbase + V::BAR_OFF + 8 * (B_SFULL + sb));
      }
    }
    __syncwarp();
  } else if (ntiles > 0 && warp == kPvWarp) {
    // ================= P V issue (one thread) =================
    // PV(k) follows QK(k): its P was made from the scores QK(k) wrote. The
    // operand buffer's K and V are free once PV(k) completes.
    if (lane == 0) {
      constexpr uint32_t idesc_pv = tc::f16_idesc(VM, D, 0, true);
      int u = unit_of(Pt, U, g0), prev_u = -1, seg = 0;
      for (int k = 0; k < ntiles; ++k) {
        const int g = g0 + k;
        while (Pt[u + 1] <= g) ++u;
        const bool seg_start = u != prev_u;
        const bool seg_end = k == ntiles - 1 || g + 1 >= Pt[u + 1];
        if (!W.wait(B_PFULL + k % NSB, (k / NSB) & 1)) break;
        if (seg_start && seg > 0 && !W.wait(B_OFREE, (seg - 1) & 1)) break;
        tc::fence_after();
        const uint32_t vbase = sbase + V::WB_OFF + (k % NWB) * V::ST_BYTES + V::KT_BYTES;
#pragma unroll
        for (int kk = 0; kk < VNK / 16; ++kk) {
          const uint64_t db = tc::sw128_desc(vbase + kk * 2048, V::KT_REG, 1024);
          tc::mma_ts(tmem + V::O_COL, tmem + V::S_COL + (k % NSB) * V::S_BUF + kk * 8, db, idesc_pv,
                     !seg_start || kk > 0);
        }
        tc::commit(sbase + V::BAR_OFF + 8 * (B_PVDONE + (k & 1)));
        tc::commit(sbase + V::BAR_OFF + 8 * (B_SDONE + k % NSB));
        tc::commit(sbase + V::BAR_OFF + 8 * (B_WFREE + k % NWB));
        if (seg_end) ++seg;
        prev_u = u;
      }
    }
    __syncwarp();
  } else if (ntiles > 0 && warp < kSoftWarps) {
    // ================= softmax: thread t owns row t =================
    pdl_wait();  // q rotated by the prologue
    pdl_trigger();
    const int t = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
    int u = unit_of(Pt, U, g0), prev_u = -1, seg = 0;
    float m_ref = -INFINITY, l = 0.f;
    for (int k = 0; k < ntiles; ++k) {
      const int g = g0 + k;
      while (Pt[u + 1] <= g) ++u;
      const bool seg_start = u != prev_u;
      const bool seg_end = k == ntiles - 1 || g + 1 >= Pt[u + 1];
      if (seg_start) {
        // this unit's q rows as fp16 pairs into tensor memory (the QK MMAs'
        // A operand; the previous unit's QKs are done: its last scores were read)
        const int s = u / Hkv, j = u - s * Hkv;
        const uint16_t* src = nullptr;
        if (t < R) {
          const int gq = t / T, i = t - gq * T;
          src = a.qhat16 + ((static_cast<int64_t>(s) * T + i) * Hq + j * G + gq) * D;
        }
#pragma unroll 1
        for (int c32 = 0; c32 < D / 64; ++c32) {
          uint32_t qv[32];  // fp16 pairs, the lower dim in the low half
#pragma unroll
          for (int x = 0; x < 32; x += 4) {
            uint4 y = make_uint4(0u, 0u, 0u, 0u);
            if (src) y = *reinterpret_cast<const uint4*>(src + 64 * c32 + 2 * x);
            qv[x] = y.x;
            qv[x + 1] = y.y;
            qv[x + 2] = y.z;
            qv[x + 3] = y.w;
          }
          tc::st32(tmem + lane_off + V::Q_COL + 32 * c32, qv);
        }
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sbase + V::BAR_OFF + 8 * B_QREADY);
        m_ref = -INFINITY;
        l = 0.f;
      }
      const int sb = k % NSB;
      if (!__all_sync(0xffffffffu, W.wait(B_SFULL + sb, (k / NSB) & 1))) break;
      tc::fence_after();
      uint32_t sr[VNK];
      static_assert(VNK == 32, "one 32-column score read per row");
      tc::ld32(tmem + lane_off + V::S_COL + sb * V::S_BUF, sr);
      tc::wait_ld();
      const int nvalid = min(VNK, Nn[u] - (g - Pt[u]) * VNK);
      float tmax = -INFINITY;
#pragma unroll
      for (int x = 0; x < VNK; ++x) {
        const float sx = x < nvalid ? __uint_as_float(sr[x]) : -INFINITY;
        sr[x] = __float_as_uint(sx);
        tmax = fmaxf(tmax, sx);
      }
      if (m_ref == -INFINITY) {
        m_ref = tmax;
      } else {
        const bool need = tmax > m_ref + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
          // rescale this warp's rows of O once the last PV has landed
          if (!__all_sync(0xffffffffu, W.wait(B_PVDONE + ((k - 1) & 1), ((k - 1) >> 1) & 1))) break;
          tc::fence_after();
          const float f = need ? exp2_fast(m_ref - tmax) : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tc::ld32(tmem + lane_off + V::O_COL + cc * 32, o);
            tc::wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * f);
            tc::st32(tmem + lane_off + V::O_COL + cc * 32, o);
          }
          tc::wait_st();
          if (need) {
            l *= f;
            m_ref = tmax;
          }
        }
      }
      // probabilities in fp16; the row sum uses the same rounded values
      uint32_t ph[VNK / 2];
      float lsum = 0.f;
#pragma unroll
      for (int x = 0; x < VNK / 2; ++x) {
        const float p0 = exp2_fast(__uint_as_float(sr[2 * x]) - m_ref);
        const float p1 = exp2_fast(__uint_as_float(sr[2 * x + 1]) - m_ref);
        const __half2 h = __floats2half2_rn(p0, p1);
        lsum += __low2float(h) + __high2float(h);
        ph[x] = *reinterpret_cast<const uint32_t*>(&h);
      }
      l += lsum;
      // row t of P (fp16 pairs) over this tile's scores, where PV reads its A
      // operand (the scores were read above; the PV NSB tiles back that read
      // this buffer's P completed before QK(k) was issued)
      tc::st16(tmem + lane_off + V::S_COL + sb * V::S_BUF, ph);
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sbase + V::BAR_OFF + 8 * (B_PFULL + sb));
      if (seg_end) {
        if (!__all_sync(0xffffffffu, W.wait(B_PVDONE + (k & 1), (k >> 1) & 1))) break;
        tc::fence_after();
        const int slot = seg == 0 ? cta : NC + u;
        float* dst = a.part + (static_cast<int64_t>(slot) * R + t) * row_stride<D>();
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tc::ld32(tmem + lane_off + V::O_COL + cc * 32, o);
          tc::wait_ld();
          if (t < R) {
#pragma unroll
            for (int x = 0; x < 32; x += 4)
              *reinterpret_cast<float4*>(dst + cc * 32 + x) =
                  make_float4(__uint_as_float(o[x]), __uint_as_float(o[x + 1]), __uint_as_float(o[x + 2]),
                              __uint_as_float(o[x + 3]));
          }
        }
        if (t < R) {
          dst[D] = m_ref;
          dst[D + 1] = l;
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sbase + V::BAR_OFF + 8 * B_OFREE);
        ++seg;
      }
      prev_u = u;
    }
  }

  tc::fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after();
    tc::dealloc(tmem, V::TMEM_COLS);
  }
  // The combine may begin once every CTA of this pass has triggered, and each
  // one does so only after the prologue has completed: so the combine reads the
  // rotated q and window keys before waiting for this pass.
  pdl_wait();
  pdl_trigger();
}

// ---------------------------------------------------------------- combine

template <int D>
__global__ void __launch_bounds__(256) verify_combine_kernel(const VerifyCombineArgs a) {
  constexpr int EPL = D / 32;  // dims per lane
  __shared__ int par_s[16];
  __shared__ int path_s[16];
  __shared__ int npath_s;
  const int i = blockIdx.x, j = blockIdx.y, s = blockIdx.z;
  const int g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.G, T = a.T, Hkv = a.Hkv, Hq = Hkv * G, R = G * T, h = j * G + g;
  const int64_t tok = static_cast<int64_t>(s) * T + i;
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
  if (a.gate) sig = 1.f / (1.f + expf(-bf16_to_f32(a.gate[tok * Hq + h])));
  int n = c.seq_len[s];
  const int cap = min(a.max_len, c.bt_stride * c.P);
  n = n < 0 ? 0 : (n > cap ? cap : n);
  int64_t wb_off = -1;
  if (a.write_back && g == 0) {
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
  float sw[16];
  float M = -INFINITY;
#pragma unroll 1
  for (int p = 0; p < np; ++p) {
    const uint16_t* kp = a.khat + ((static_cast<int64_t>(s) * T + path_s[p]) * Hkv + j) * D + lane * EPL;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; e += 2) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(kp + e);
      dot = fmaf(q[e], bf16_lo(w), dot);
      dot = fmaf(q[e + 1], bf16_hi(w), dot);
    }
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, w);
    sw[p] = dot;
    M = fmaxf(M, dot);
  }
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float L = 0.f;  // relative to M
#pragma unroll 1
  for (int p = 0; p < np; ++p) {
    const float w = exp2_fast(sw[p] - M);
    L += w;
    const uint16_t* vp = a.v + ((static_cast<int64_t>(s) * T + path_s[p]) * Hkv + j) * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; e += 2) {
      const uint32_t x = *reinterpret_cast<const uint32_t*>(vp + e);
      acc[e] = fmaf(w, bf16_lo(x), acc[e]);
      acc[e + 1] = fmaf(w, bf16_hi(x), acc[e + 1]);
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
  float* dst = a.out + (tok * Hq + h) * D + lane * EPL;
#pragma unroll
  for (int e = 0; e < EPL; e += 4)
    *reinterpret_cast<float4*>(dst + e) =
        make_float4(acc[e] * scale, acc[e + 1] * scale, acc[e + 2] * scale, acc[e + 3] * scale);

  // ---- write-back of this node's entry at token index prefix_len + i
  if (wb_off >= 0) {
    const uint16_t* kh = a.khat + (tok * Hkv + j) * D + lane * EPL;
    const uint16_t* vv = a.v + (tok * Hkv + j) * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; e += 4) {
      *reinterpret_cast<uint2*>(c.k + wb_off + lane * EPL + e) = *reinterpret_cast<const uint2*>(kh + e);
      *reinterpret_cast<uint2*>(c.v + wb_off + lane * EPL + e) = *reinterpret_cast<const uint2*>(vv + e);
    }
  }
}

template <int D>
cudaError_t verify_split_launch(const VerifySplitArgs& a, cudaStream_t s) {
  using V = VGeo<D>;
  static std::atomic<uint64_t> opted{0};
  const cudaError_t e = opt_in_smem(verify_split_kernel<D>, V::SMEM, opted);
  if (e != cudaSuccess) return e;
  return launch_pdl(verify_split_kernel<D>, dim3(a.ctas), dim3(kVThreads), V::SMEM, s, a);
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
