// Internal interface between the host planner (dattn.cu) and the kernel
// translation units. Not part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cmath>
#include <utility>

namespace dattn {

// RoPE angle step of pair i of an r-dim rotation with base theta, in 64-bit
// fixed-point turns per position: rint(2^64 * theta^(-2i/r) / 2pi), the
// frequency and the division by 2pi each rounded to fp64.
inline uint64_t rope_phase_step(double theta, int r, int i) {
  const double inv_freq = std::pow(theta, -static_cast<double>(2 * i) / static_cast<double>(r));
  return static_cast<uint64_t>(std::llrint(std::ldexp(inv_freq / 6.283185307179586, 64)));
}

// Sticky device error bits (see dattn_get_error).
enum : int { ERR_INDEX = 1, ERR_TIMEOUT = 2, ERR_LENGTH = 4, ERR_RANGE = 8 };

// Limit of a bounded device wait unless the handle sets another (2 s).
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
// Testing aid (dattn_debug_config): the decode kernel's helper warp withholds
// the first unit's rotated query, so the streaming warps' waits run out.
constexpr int kDebugWithholdQ = 1;

// One layer's cache as the kernels see it.
struct CacheView {
  uint16_t* k;                 // ring [n_rows, Hkv, R, D] / paged [pages, Hkv, P, D]
  uint16_t* v;
  int paged;                   // 0 = ring, 1 = paged
  int n_rows;                  // ring rows or pages in the pool
  int R;                       // ring slots
  int P;                       // page size
  const int32_t* ring_head;    // [B]
  const int32_t* ring_count;   // [B]
  const int32_t* stream_rows;  // [B] or null
  const int32_t* block_table;  // [B, bt_stride]
  int bt_stride;
  const int32_t* seq_len;      // [B]
};

// RoPE prologue: rotates q (fp32 out, pre-scaled) and k (bf16 entry out) of
// `rows` token rows. Decode: row = stream, position pos[row]. Verify: row =
// s * T + i, position prefix_len[s] + depth(i) from the parent array.
struct RopeArgs {
  int rows;
  int Hq, Hkv, D, r;
  const uint16_t* q;           // [rows, Hq, D]
  const uint16_t* k;           // [rows, Hkv, D]
  const int32_t* pos;          // [rows] (decode) or null
  const int32_t* prefix_len;   // [rows / T] (verify) or null
  const int32_t* parent;       // [rows] (verify) or null
  int T;
  const uint64_t* rope_step;   // [r / 2] phase steps (rope_phase_step)
  float q_scale;               // log2(e) / sqrt(D)
  float* qhat;                 // [rows, Hq, D]
  uint16_t* qhl;               // [2][qhl_rows, Hq, D]: the same values as bf16 hi, then the
                               // bf16 rounding of what is left (lo), or null
  int qhl_rows;                // rows of one plane of qhl (its capacity)
  uint16_t* khat;              // [rows, Hkv, D]
  int* err;
  const uint16_t* q_norm;      // [D] QK-norm weights, or null
  const uint16_t* k_norm;
  double norm_eps;
  // Row r = s * T + i reads the caller's q/k row s * in_T + row0 + i (a
  // prefill chunk of a longer array; rows past in_T read as zero). Verify:
  // in_T = T, row0 = 0.
  int in_T, row0;
};

// Query heads of a KV group as the decode kernel lays them out: 4 (G <= 4)
// or 8 (G <= 8); 0 for a group size with no compiled kernel.
inline int decode_group_pad(int G) { return G <= 0 ? 0 : (G <= 4 ? 4 : (G <= 8 ? 8 : 0)); }

// One decode call (RoPE of the new token, the pass over the cached keys, the
// join in score space, gate, store, write-back) as one launch. Stream-K: the
// grid cuts the concatenated tiles of all (stream, KV head) units into equal
// ranges. Partial slot of a segment: the CTA index for the first segment of a
// CTA's range, gridDim + unit for any later one; the CTA that finishes a
// unit's last segment (per-unit counter) combines the unit.
struct DecodeArgs {
  CUtensorMap tmap_k;          // the layer's K cache as a 2D [rows, D] bf16 tensor
  CUtensorMap tmap_v;          // (encode_cache_maps)
  CacheView c;
  int B, Hkv, G;
  int max_len;                 // host bound on cached length (paged)
  const uint16_t* q;           // [B, Hq, D]
  const uint16_t* k_new;       // [B, Hkv, D]
  const uint16_t* v_new;       // [B, Hkv, D]
  const uint16_t* gate;        // [B, Hq] or null
  const int32_t* pos;          // [B]
  const uint64_t* rope_step;   // [r / 2] phase steps (rope_phase_step)
  int r;
  float q_scale;               // log2(e) / sqrt(D)
  float* out;                  // [B, Hq, D]
  int write_back;
  float* part;                 // [ctas + B*Hkv][GP*(D+2)]: o[GP][D], m[GP], l[GP]
                               // (GP = decode_group_pad(G))
  int* counters;               // [B*Hkv] finished segments, then [ctas] group counters; zero between calls
  int* err;
  int early;                   // nonzero: the preceding launch on the stream writes
                               // no part of this cache, so the first cache loads may
                               // start before it completes
  int unit_cost;               // fixed cost of one segment of a unit, in stage tiles
                               // (set by launch_decode)
  uint64_t wait_ns;            // limit of every bounded wait (0 = kDefaultWaitNs)
  int debug_flags;             // kDebugWithholdQ: see dattn_debug_config
  const uint16_t* q_norm;      // [D] QK-norm weights of the queries, or null
  const uint16_t* k_norm;      // [D] of the new key, or null
  double norm_eps;
  // E4M3 cache (the pools hold bytes; k, v of CacheView are byte arrays):
  // cached value = e4m3 * scale. q_scale then includes k_scale.
  int f8;
  float k_scale, v_scale;
};

struct AppendArgs {
  CacheView c;
  int B, Tmax, Hkv, D, r;
  const int32_t* start_index;
  const int32_t* start_pos;
  const int32_t* count;
  const uint16_t* k;           // [B, Tmax, Hkv, D]
  const uint16_t* v;
  int rotate;
  const uint64_t* rope_step;   // [r / 2]
  int* err;
  const uint16_t* k_norm;      // [D] QK-norm weights of the keys (with rotate), or null
  double norm_eps;
  // source rows: b * in_T + row0 + t of k/v (in_T = Tmax, row0 = 0 but for
  // prefill chunks)
  int in_T, row0;
  // E4M3 pools: entries stored as the E4M3 bytes nearest entry / k_scale
  // (K) and v / v_scale (V)
  int f8;
  float k_scale, v_scale;
  // commit of verify paths: token t of row b is source row gather[b * Tmax + t]
  // of k/v ([B, Tmax, Hkv, D]), and the row's first count[b] entries of gather
  // must form a path from a root under parent [B, Tmax]; null for a plain append
  const int32_t* gather;
  const int32_t* parent;
};

// Tensor-core pass of tree verify over each stream's paged prefix (stream-K
// over (stream, KV head) units and their 128-key tiles; the G*T rows of a
// unit are one 128-row MMA tile).
// Partial slot layout: [ctas + S*Hkv][G*T rows][D + 4] fp32 (o[D], m, l, pad),
// row g * T + i for query head g of the group and tree node i.
struct VerifySplitArgs {
  CUtensorMap tmap_k;          // the layer's K pool as [rows, D] bf16, boxes of 16 rows x 64 dims
  CUtensorMap tmap_v;          // its V pool as (64 dims, rows, D/64 regions), boxes of (64, 16, D/64)
  CUtensorMap tmap_q;          // q hi/lo as (D, Hq, S*T, 2) bf16, boxes of (64, G, T, 1)
  CacheView c;                 // paged (page size a multiple of 16; seq_len = prefix lengths)
                               // or ring (all R slots scanned, the valid ones kept)
  int S, T, Hkv, G;
  const int32_t* parent;       // [S, T] (ring layers: a row's depth sets how many of the
                               // oldest entries its path pushed out)
  const uint16_t* qhl;         // [2][qhl_rows, Hq, D]: q as bf16 hi (the first plane) and lo
  int ctas;
  int max_len;
  float* part;
  int* tiles;                  // out, U = S*Hkv: [U + 1] tile prefix over units, then per
                               // unit the first CTA of its span [U], the span's length [U]
                               // and the partial slot of its first segment [U]
  int* err;
};

// Ragged prefill in chunks of Tc tokens: the cache state a chunk starts from
// (the caller's plus the min(count, row0) tokens of earlier chunks) and the
// chunk's token count and root position, per stream, into scratch arrays.
struct PrefillMetaArgs {
  CacheView c;                 // the caller's cache metadata
  const int32_t* count;        // [S] new tokens of each stream (0..Tmax)
  const int32_t* start_pos;    // [S] position of each stream's token 0
  int S, Tmax, row0, Tc;
  int32_t* seq_c;              // paged: seq_len + m
  int32_t* head_c;             // ring: (head + m) mod R
  int32_t* cnt_c;              // ring: min(count + m, R)
  int32_t* pos_c;              // start_pos + row0
  int32_t* n_c;                // tokens of this chunk: clamp(count - row0, 0, Tc)
  int32_t* chain;              // [S, Tc] chain-tree parents: i - 1
  int* err;
};
cudaError_t launch_prefill_meta(const PrefillMetaArgs& a, cudaStream_t s);

// Tree-window join: merge the prefix segments of each row, score the row's
// path in the window (its ancestors and itself), gate, store, write back.
struct VerifyCombineArgs {
  CacheView c;
  int S, T, Hkv, G;
  int split_ctas;
  const int* tiles;            // written by the split pass (VerifySplitArgs::tiles)
  int max_len;
  const float* qhat;           // [S*T, Hq, D]
  const uint16_t* khat;        // [S*T, Hkv, D] rotated window keys (bf16 entries)
  const uint16_t* v;           // [S, T, Hkv, D]
  const int32_t* parent;       // [S, T]
  const uint16_t* gate;        // [S, T, Hq] or null
  const float* part;
  float* out;                  // [S, T, Hq, D]
  int write_back;
  int* err;
  // caller rows of v, gate and out: s * in_T + row0 + i (see RopeArgs); with
  // rows_valid, only rows i < rows_valid[s] are stored (prefill chunks)
  int in_T, row0;
  const int32_t* rows_valid;
};

// Decode grid: every resident CTA (`resident` on the whole GPU), but at
// least 4 stage tiles (one per streaming warp) per CTA for the largest amount
// of work the call may have: `units` units of up to `n_max` keys each.
inline int plan_decode_ctas(int resident, int units, int n_max, int tile_keys) {
  const int64_t tiles = static_cast<int64_t>(units) * ((n_max + tile_keys - 1) / tile_keys);
  int64_t ctas = (tiles + 3) / 4;
  if (ctas > resident) ctas = resident;
  if (ctas < 1) ctas = 1;
  return static_cast<int>(ctas);
}

// Each returns cudaErrorNotSupported for a shape with no compiled kernel.
cudaError_t launch_rope(const RopeArgs& a, cudaStream_t s, bool pdl = true);
// Decode with `ctas` CTAs (at most decode_ctas_per_sm per SM). With pdl the
// launch is a programmatic dependent of the previous one on the stream;
// without, it starts once everything before it on the stream has completed.
cudaError_t launch_decode(const DecodeArgs& a, int D, int ctas, cudaStream_t s, bool pdl = true);
// Tensor maps of a cache's K and V for the decode kernel over its [n_rows *
// Hkv * (R or P), D] bf16 rows, 128-byte swizzle: at D = 128 seen as (64 dims,
// row, 2 regions) with one box per 16-row group; at D = 256 as [rows, D] with
// boxes of 16 rows x 64 dims.
cudaError_t encode_cache_maps(const CacheView& c, int Hkv, int D, CUtensorMap* k, CUtensorMap* v, bool f8 = false);
cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);
// decode over an E4M3 cache (decode_fp8.cu); GP = decode_group_pad(G)
cudaError_t launch_decode_fp8(const DecodeArgs& a, int D, int GP, int ctas, cudaStream_t s, bool pdl);
cudaError_t launch_verify_split(const VerifySplitArgs& a, int D, cudaStream_t s);
cudaError_t launch_verify_combine(const VerifyCombineArgs& a, int D, cudaStream_t s);
// Keys per tile of the verify pass and its largest unit count.
constexpr int kVerifyTileKeys = 128;
// Fixed cost of one unit segment of the verify pass's split, in tiles.
constexpr int kVerifySegmentCost = 2;
constexpr int kVerifyMaxUnits = 512;
// Most rows (G * T) of a verify unit: one 128-row MMA tile.
constexpr int kVerifyMaxRows = 128;
// Tensor maps of the verify pass: the K pool as [rows, D] bf16 with boxes of
// 16 rows x 64 dims, the V pool as (64, rows, D/64) with boxes of (64, 16,
// D/64) (a 16-row group, all dims), and q hi/lo (qhl, planes of qhl_rows
// rows) as (D, Hq, S*T, 2) bf16 with boxes of (64, G, T, 1); all 128-byte
// swizzled.
cudaError_t encode_verify_maps(const CacheView& c, int Hkv, int D, const uint16_t* qhl, int qhl_rows, int Hq,
                               int G, int S, int T, CUtensorMap* k, CUtensorMap* v, CUtensorMap* q);

// Resident CTAs per SM of the decode kernel for (D, G) (0 if unsupported).
int decode_ctas_per_sm(int D, int G);
// Keys per stage tile of the decode kernel for (D, G).
int decode_tile_keys(int D, int G, bool f8 = false);
// Largest number of (stream, KV head) units of one decode call.
int decode_max_units();

// Launch order per stream, for early cache reads. A kernel launched with
// programmatic stream serialization may run while the launch before it on the
// stream finishes; that launch is the only one that can still be writing.
// True when the last launch recorded on `stream` writes into the cache whose
// K array is `cache_k`.
bool prev_launch_writes(void* stream, const void* cache_k);
// Record a launch made on `stream` that writes into the cache with K array
// `cache_k` (null: writes no cache).
void record_launch(void* stream, const void* cache_k);

// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device (`done` holds one bit per device id below 64; the
// call is idempotent, so racing threads at worst repeat it).
template <typename Kernel>
cudaError_t opt_in_smem(Kernel kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
  if (bit != 0ull && (done.load(std::memory_order_acquire) & bit) != 0ull) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0ull) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Launch with programmatic stream serialization: the kernel may begin while
// its predecessor in the stream finishes; every kernel here waits on the
// predecessor (griddepcontrol.wait) before it touches the predecessor's output.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace dattn
