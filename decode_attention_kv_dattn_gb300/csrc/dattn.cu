// Host side of the dattn C ABI: argument checks, the workspace, the split
// plan and the launches of each call.
//
// A decode call is one kernel launch (decode_kernel): RoPE of the new token,
// the pass over the cached keys, the join in score space, the gate, the fp32
// store and the write-back of the new entry, which comes after every read of
// the cache (when a ring is full the new entry takes the oldest slot). A
// verify call is three launches (the RoPE prologue, the tensor-core pass over
// the prefix, the combine with the tree part), each a programmatic dependent
// of the one before.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include <mutex>
#include <unordered_map>

#include "dattn.h"
#include "kernels.h"

using namespace dattn;

namespace dattn {

namespace {
std::mutex g_order_mutex;
std::unordered_map<void*, const void*> g_last_written;  // stream -> cache K written by its last launch
}  // namespace

bool prev_launch_writes(void* stream, const void* cache_k) {
  std::lock_guard<std::mutex> lock(g_order_mutex);
  const auto it = g_last_written.find(stream);
  return it != g_last_written.end() && it->second == cache_k;
}

void record_launch(void* stream, const void* cache_k) {
  std::lock_guard<std::mutex> lock(g_order_mutex);
  g_last_written[stream] = cache_k;
}

}  // namespace dattn

struct dattn_handle {
  int device = 0;
  int Hq = 0, Hkv = 0, D = 0, G = 0, GP = 0;
  int max_streams = 0, max_context = 0, max_verify_rows = 0;
  std::vector<dattn_layer_config> layers;
  std::vector<uint64_t*> rope_step;  // device, per layer ([r/2] phase steps or null)
  std::vector<uint16_t*> q_norm, k_norm;  // device, per layer ([D] QK-norm weights or null)
  int num_sms = 0;
  int decode_resident = 0;  // resident decode CTAs on the whole GPU
  size_t part_units = 0;    // capacity of the decode partials, in segment slots
  // Decode workspace, two halves used by alternate calls (a call may run while
  // the one before it finishes): partials [part_units][GP][D+2] and finished
  // segments per (stream, KV head), zero between calls.
  float* part[2] = {nullptr, nullptr};
  int* counters[2] = {nullptr, nullptr};
  unsigned decode_calls = 0;
  float* qhat = nullptr;    // verify: rotated q of the window rows
  uint16_t* qhl = nullptr;  // the same as bf16 hi and lo planes (the tensor-core pass's operand)
  int qhl_rows = 0;         // rows of one plane
  int* tiles = nullptr;     // verify: tile prefix over units, from its split pass
  uint16_t* khat = nullptr; // verify: rotated window keys
  float* vpart = nullptr;   // verify partials: [sms + units][G*T][D+4]
  int32_t* chain = nullptr;    // prefill: chain-tree parents of a chunk, [S][Tc]
  int32_t* pmeta = nullptr;    // prefill chunk state: 5 arrays of [max_streams]
  size_t vpart_slots = 0;
  int* err = nullptr;
  uint64_t wait_ns = kDefaultWaitNs;  // limit of the kernels' bounded waits
  int debug_flags = 0;                // dattn_debug_config
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }


// Make `dev` current for the duration of a call and restore the caller's.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      return;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// With DATTN_VERBOSE set in the environment, a failed launch names its CUDA
// error on stderr (the status code alone says only DATTN_ECUDA).
int cuda_status(cudaError_t e, const char* what = "launch") {
  if (e == cudaSuccess) return DATTN_OK;
  static const bool verbose = std::getenv("DATTN_VERBOSE") != nullptr;
  if (verbose) std::fprintf(stderr, "dattn: %s: %s (%s)\n", what, cudaGetErrorName(e), cudaGetErrorString(e));
  if (e == cudaErrorNotSupported) {
    cudaGetLastError();
    return DATTN_EUNSUPPORTED;
  }
  return DATTN_ECUDA;
}

CacheView make_view(const dattn_handle* h, const dattn_layer_config& L, const dattn_cache* c) {
  CacheView v{};
  v.k = static_cast<uint16_t*>(c->k);
  v.v = static_cast<uint16_t*>(c->v);
  v.paged = L.cache_kind == DATTN_CACHE_PAGED;
  v.n_rows = c->n_rows;
  v.R = L.ring_slots;
  v.P = L.page_size;
  v.ring_head = c->ring_head;
  v.ring_count = c->ring_count;
  v.stream_rows = c->stream_rows;
  v.block_table = c->block_table;
  v.bt_stride = c->bt_stride;
  v.seq_len = c->seq_len;
  (void)h;
  return v;
}

int check_cache(const dattn_layer_config& L, const dattn_cache* c) {
  if (!c || !c->k || !c->v || c->n_rows <= 0) return DATTN_EINVAL;
  if (!aligned16(c->k) || !aligned16(c->v)) return DATTN_EINVAL;
  if (L.cache_kind == DATTN_CACHE_RING) {
    if (!c->ring_head || !c->ring_count) return DATTN_EINVAL;
  } else {
    if (!c->block_table || !c->seq_len || c->bt_stride <= 0) return DATTN_EINVAL;
  }
  return DATTN_OK;
}

// One pass of the verify pipeline (three launches): the RoPE prologue, the
// tensor-core pass over the cache and the tree-window join. Shared by
// dattn_verify and by the chunks of dattn_prefill.
struct VerifyRound {
  CacheView c;
  int S, T, n_max;
  const uint16_t *q, *k, *v, *gate;
  const int32_t* parent;
  const int32_t* pos;          // [S] root positions
  float* out;
  int write_back;
  int in_T, row0;              // caller rows: s * in_T + row0 + i
  const int32_t* rows_valid;   // or null
  bool after_plain_launch;     // the launch before wrote what the prologue reads early
};

int verify_round(dattn_t* h, int layer, const VerifyRound& r, cudaStream_t s) {
  const dattn_layer_config& L = h->layers[layer];
  VerifySplitArgs va{};
  va.c = r.c;
  // one CTA per SM, at least one tile each for the largest prefix this call may have
  const int64_t tiles = static_cast<int64_t>(r.S) * h->Hkv * ((r.n_max + kVerifyTileKeys - 1) / kVerifyTileKeys);
  int64_t ctas = tiles;
  if (ctas > h->num_sms) ctas = h->num_sms;
  if (ctas < 1) ctas = 1;
  va.S = r.S;
  va.T = r.T;
  va.Hkv = h->Hkv;
  va.G = h->G;
  va.parent = r.parent;
  va.qhl = h->qhl;
  va.ctas = static_cast<int>(ctas);
  va.max_len = r.n_max;
  if (encode_verify_maps(va.c, h->Hkv, h->D, h->qhl, h->qhl_rows, h->Hq, h->G, r.S, r.T, &va.tmap_k, &va.tmap_v,
                         &va.tmap_q) != cudaSuccess)
    return DATTN_EUNSUPPORTED;

  RopeArgs ra{};
  ra.rows = r.S * r.T;
  ra.Hq = h->Hq;
  ra.Hkv = h->Hkv;
  ra.D = h->D;
  ra.r = L.rotary_dim;
  ra.q = r.q;
  ra.k = r.k;
  ra.prefix_len = r.pos;
  ra.parent = r.parent;
  ra.T = r.T;
  ra.rope_step = h->rope_step[layer];
  ra.q_scale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(h->D)));
  ra.qhat = h->qhat;
  ra.qhl = h->qhl;
  ra.qhl_rows = h->qhl_rows;
  ra.khat = h->khat;
  ra.err = h->err;
  ra.q_norm = h->q_norm[layer];
  ra.k_norm = h->k_norm[layer];
  ra.norm_eps = L.norm_eps;
  ra.in_T = r.in_T;
  ra.row0 = r.row0;
  int rc = cuda_status(launch_rope(ra, s, !r.after_plain_launch), "verify prologue");
  if (rc != DATTN_OK) return rc;

  va.part = h->vpart;
  va.tiles = h->tiles;
  va.err = h->err;
  rc = cuda_status(launch_verify_split(va, h->D, s), "verify pass");
  if (rc != DATTN_OK) return rc;

  VerifyCombineArgs vc{};
  vc.c = va.c;
  vc.S = r.S;
  vc.T = r.T;
  vc.Hkv = h->Hkv;
  vc.G = h->G;
  vc.split_ctas = va.ctas;
  vc.tiles = h->tiles;
  vc.max_len = r.n_max;
  vc.qhat = h->qhat;
  vc.khat = h->khat;
  vc.v = r.v;
  vc.parent = r.parent;
  vc.gate = r.gate;
  vc.part = h->vpart;
  vc.out = r.out;
  vc.write_back = r.write_back;
  vc.err = h->err;
  vc.in_T = r.in_T;
  vc.row0 = r.row0;
  vc.rows_valid = r.rows_valid;
  return cuda_status(launch_verify_combine(vc, h->D, s), "verify combine");
}

}  // namespace

extern "C" {

const char* dattn_error_string(int code) {
  switch (code) {
    case DATTN_OK: return "ok";
    case DATTN_EINVAL: return "invalid argument";
    case DATTN_EXCEEDS: return "request exceeds what the handle was created for";
    case DATTN_ECUDA: return "CUDA runtime error";
    case DATTN_EINDEX: return "device metadata out of range (page id, ring slot, tree parent)";
    case DATTN_ETIMEOUT: return "a bounded device wait timed out";
    case DATTN_EUNSUPPORTED: return "shape not supported: no compiled kernel for it";
    case DATTN_ELENGTH: return "a stream is longer than the call's bound";
    case DATTN_ERANGE: return "a cached value lies outside the fp16 range the verify pass forms P V in";
    default: return "unknown dattn status";
  }
}

int dattn_create(const dattn_config* cfg, int device, dattn_t** out) {
  if (!cfg || !out) return DATTN_EINVAL;
  *out = nullptr;
  const int Hq = cfg->num_q_heads, Hkv = cfg->num_kv_heads, D = cfg->head_dim;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return DATTN_EINVAL;
  if (D != 128 && D != 256) return DATTN_EUNSUPPORTED;
  const int G = Hq / Hkv;
  if (decode_group_pad(G) == 0) return DATTN_EUNSUPPORTED;
  if (cfg->max_streams <= 0 || cfg->max_context < 0 || cfg->num_layers <= 0 || !cfg->layers)
    return DATTN_EINVAL;
  if (cfg->max_verify_rows < 0 || cfg->max_verify_rows > 16) return DATTN_EINVAL;
  for (int l = 0; l < cfg->num_layers; ++l) {
    const dattn_layer_config& L = cfg->layers[l];
    if (L.cache_kind == DATTN_CACHE_RING) {
      if (L.ring_slots <= 0) return DATTN_EINVAL;
    } else if (L.cache_kind == DATTN_CACHE_PAGED) {
      if (L.page_size <= 0) return DATTN_EINVAL;
    } else {
      return DATTN_EINVAL;
    }
    if (L.rotary_dim < 0 || L.rotary_dim > D || L.rotary_dim % 2) return DATTN_EINVAL;
    if (L.rotary_dim > 0 && !(L.rope_theta > 0.0)) return DATTN_EINVAL;
    if ((L.q_norm_weight || L.k_norm_weight) && !(L.norm_eps >= 0.0)) return DATTN_EINVAL;
    if (L.kv_format != DATTN_KV_BF16 && L.kv_format != DATTN_KV_E4M3) return DATTN_EINVAL;
    if (L.kv_format == DATTN_KV_E4M3 &&
        !(L.k_scale > 0.f && L.v_scale > 0.f && std::isfinite(L.k_scale) && std::isfinite(L.v_scale)))
      return DATTN_EINVAL;
  }
  DeviceGuard guard(device);
  if (!guard.ok) return DATTN_ECUDA;

  dattn_handle* h = new (std::nothrow) dattn_handle();
  if (!h) return DATTN_ECUDA;
  h->device = device;
  h->Hq = Hq;
  h->Hkv = Hkv;
  h->D = D;
  h->G = G;
  h->GP = decode_group_pad(G);
  h->max_streams = cfg->max_streams;
  h->max_context = cfg->max_context;
  h->max_verify_rows = cfg->max_verify_rows;
  h->layers.assign(cfg->layers, cfg->layers + cfg->num_layers);

  auto fail = [&](int code) {
    dattn_destroy(h);
    return code;
  };
  if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return fail(DATTN_ECUDA);
  h->decode_resident = h->num_sms * decode_ctas_per_sm(D, G);
  if (h->decode_resident <= 0) return fail(DATTN_EUNSUPPORTED);

  // RoPE phase steps (fixed-point turns per position), one table per layer
  for (const dattn_layer_config& L : h->layers) {
    uint64_t* dev = nullptr;
    if (L.rotary_dim > 0) {
      // whole 16-byte units: the decode kernel bulk-copies the table
      std::vector<uint64_t> f((L.rotary_dim / 2 + 1) / 2 * 2, 0);
      for (int i = 0; i < L.rotary_dim / 2; ++i) f[i] = rope_phase_step(L.rope_theta, L.rotary_dim, i);
      if (cudaMalloc(&dev, f.size() * sizeof(uint64_t)) != cudaSuccess) return fail(DATTN_ECUDA);
      h->rope_step.push_back(dev);
      if (cudaMemcpy(dev, f.data(), f.size() * sizeof(uint64_t), cudaMemcpyHostToDevice) != cudaSuccess)
        return fail(DATTN_ECUDA);
    } else {
      h->rope_step.push_back(nullptr);
    }
  }

  // QK-norm weights, one [D] copy per layer and side; the handle keeps no
  // host pointer of the caller's
  for (dattn_layer_config& L : h->layers) {
    for (int side = 0; side < 2; ++side) {
      const uint16_t* src = side == 0 ? L.q_norm_weight : L.k_norm_weight;
      uint16_t* dev = nullptr;
      if (src) {
        if (cudaMalloc(&dev, D * sizeof(uint16_t)) != cudaSuccess) return fail(DATTN_ECUDA);
        (side == 0 ? h->q_norm : h->k_norm).push_back(dev);
        if (cudaMemcpy(dev, src, D * sizeof(uint16_t), cudaMemcpyHostToDevice) != cudaSuccess)
          return fail(DATTN_ECUDA);
      } else {
        (side == 0 ? h->q_norm : h->k_norm).push_back(nullptr);
      }
    }
    L.q_norm_weight = L.k_norm_weight = nullptr;
  }

  // Workspace. Rows of rotated q/k: one per stream (decode) or per verify row.
  const size_t rows = static_cast<size_t>(h->max_streams) *
                      (h->max_verify_rows > 1 ? h->max_verify_rows : 1);
  if (cudaMalloc(&h->qhat, rows * Hq * D * sizeof(float)) != cudaSuccess) return fail(DATTN_ECUDA);
  h->qhl_rows = static_cast<int>(rows);
  if (cudaMalloc(&h->qhl, 2 * rows * Hq * D * sizeof(uint16_t)) != cudaSuccess) return fail(DATTN_ECUDA);
  if (cudaMalloc(&h->khat, rows * Hkv * D * sizeof(uint16_t)) != cudaSuccess) return fail(DATTN_ECUDA);
  // Decode partials: one slot per CTA plus one per unit; per-unit counters,
  // then one per CTA (the group counters of units merged in two levels).
  if (static_cast<int64_t>(h->max_streams) * Hkv > decode_max_units()) return fail(DATTN_EUNSUPPORTED);
  h->part_units = static_cast<size_t>(h->decode_resident) + static_cast<size_t>(h->max_streams) * Hkv;
  for (int i = 0; i < 2; ++i) {
    const size_t nc = static_cast<size_t>(h->max_streams) * Hkv + static_cast<size_t>(h->decode_resident);
    if (cudaMalloc(&h->counters[i], nc * sizeof(int)) != cudaSuccess) return fail(DATTN_ECUDA);
    if (cudaMemset(h->counters[i], 0, nc * sizeof(int)) != cudaSuccess) return fail(DATTN_ECUDA);
  }
  if (cudaMalloc(&h->tiles, (4 * static_cast<size_t>(h->max_streams) * Hkv + 1) * sizeof(int)) != cudaSuccess)
    return fail(DATTN_ECUDA);
  const size_t part_floats = h->part_units * h->GP * (D + 2);
  for (int i = 0; i < 2; ++i)
    if (cudaMalloc(&h->part[i], part_floats * sizeof(float)) != cudaSuccess) return fail(DATTN_ECUDA);
  if (h->max_verify_rows > 0) {
    if (G * h->max_verify_rows > kVerifyMaxRows) return fail(DATTN_EUNSUPPORTED);
    if (static_cast<int64_t>(h->max_streams) * Hkv > kVerifyMaxUnits) return fail(DATTN_EUNSUPPORTED);
    h->vpart_slots = static_cast<size_t>(h->num_sms) + static_cast<size_t>(h->max_streams) * Hkv;
    const size_t vfloats = h->vpart_slots * G * h->max_verify_rows * (D + 4);
    if (cudaMalloc(&h->vpart, vfloats * sizeof(float)) != cudaSuccess) return fail(DATTN_ECUDA);
    // prefill: chain trees (written per chunk: parent of row i is i - 1) and
    // the chunk state
    const size_t nchain = static_cast<size_t>(h->max_streams) * h->max_verify_rows;
    if (cudaMalloc(&h->chain, nchain * sizeof(int32_t)) != cudaSuccess) return fail(DATTN_ECUDA);
    if (cudaMalloc(&h->pmeta, 5 * static_cast<size_t>(h->max_streams) * sizeof(int32_t)) != cudaSuccess)
      return fail(DATTN_ECUDA);
  }
  if (cudaMalloc(&h->err, sizeof(int)) != cudaSuccess) return fail(DATTN_ECUDA);
  if (cudaMemset(h->err, 0, sizeof(int)) != cudaSuccess) return fail(DATTN_ECUDA);
  *out = h;
  return DATTN_OK;
}

void dattn_destroy(dattn_t* h) {
  if (!h) return;
  DeviceGuard guard(h->device);
  for (uint64_t* p : h->rope_step) cudaFree(p);
  for (uint16_t* p : h->q_norm) cudaFree(p);
  for (uint16_t* p : h->k_norm) cudaFree(p);
  cudaFree(h->qhat);
  cudaFree(h->chain);
  cudaFree(h->pmeta);
  cudaFree(h->qhl);
  cudaFree(h->khat);
  for (int i = 0; i < 2; ++i) {
    cudaFree(h->part[i]);
    cudaFree(h->counters[i]);
  }
  cudaFree(h->vpart);
  cudaFree(h->tiles);
  cudaFree(h->err);
  delete h;
}

int dattn_debug_config(dattn_t* h, int flags, unsigned wait_limit_us) {
  if (!h || (flags & ~DATTN_DEBUG_WITHHOLD_Q) != 0) return DATTN_EINVAL;
  h->debug_flags = (flags & DATTN_DEBUG_WITHHOLD_Q) ? kDebugWithholdQ : 0;
  h->wait_ns = wait_limit_us ? static_cast<uint64_t>(wait_limit_us) * 1000ull : kDefaultWaitNs;
  return DATTN_OK;
}

int dattn_get_error(dattn_t* h, dattn_stream_t stream) {
  if (!h) return DATTN_EINVAL;
  DeviceGuard guard(h->device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int bits = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DATTN_ECUDA;
  if (cudaMemcpyAsync(&bits, h->err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DATTN_ECUDA;
  if (cudaMemsetAsync(h->err, 0, sizeof(int), s) != cudaSuccess) return DATTN_ECUDA;
  // a call that gave up waiting still counts its segments; clear them anyway
  for (int i = 0; i < 2 && bits; ++i)
    if (cudaMemsetAsync(h->counters[i], 0,
                        (static_cast<size_t>(h->max_streams) * h->Hkv + h->decode_resident) * sizeof(int),
                        s) != cudaSuccess)
      return DATTN_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DATTN_ECUDA;
  if (bits & ERR_TIMEOUT) return DATTN_ETIMEOUT;
  if (bits & ERR_INDEX) return DATTN_EINDEX;
  if (bits & ERR_RANGE) return DATTN_ERANGE;
  if (bits & ERR_LENGTH) return DATTN_ELENGTH;
  return DATTN_OK;
}

int dattn_append_kv(dattn_t* h, int layer, const dattn_cache* cache, int num_streams,
                    int max_tokens, const int32_t* start_index, const int32_t* start_pos,
                    const int32_t* count, const void* k, const void* v, int rotate,
                    dattn_stream_t stream) {
  if (!h || layer < 0 || layer >= static_cast<int>(h->layers.size())) return DATTN_EINVAL;
  const dattn_layer_config& L = h->layers[layer];
  int rc = check_cache(L, cache);
  if (rc != DATTN_OK) return rc;
  if (num_streams <= 0 || max_tokens < 0 || !start_index || !count || !k || !v) return DATTN_EINVAL;
  if (rotate && L.rotary_dim > 0 && !start_pos) return DATTN_EINVAL;
  if (!aligned16(k) || !aligned16(v)) return DATTN_EINVAL;
  if (max_tokens == 0) return DATTN_OK;
  if (max_tokens > 65535) return DATTN_EXCEEDS;
  DeviceGuard guard(h->device);
  if (!guard.ok) return DATTN_ECUDA;
  AppendArgs a{};
  a.c = make_view(h, L, cache);
  a.B = num_streams;
  a.Tmax = max_tokens;
  a.Hkv = h->Hkv;
  a.D = h->D;
  a.r = L.rotary_dim;
  a.start_index = start_index;
  a.start_pos = start_pos;
  a.count = count;
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.rotate = rotate;
  a.rope_step = h->rope_step[layer];
  a.err = h->err;
  a.k_norm = h->k_norm[layer];
  a.norm_eps = L.norm_eps;
  a.in_T = max_tokens;
  a.f8 = L.kv_format == DATTN_KV_E4M3;
  a.k_scale = L.k_scale;
  a.v_scale = L.v_scale;
  rc = cuda_status(launch_append(a, reinterpret_cast<cudaStream_t>(stream)), "append");
  if (rc == DATTN_OK) record_launch(stream, cache->k);
  return rc;
}

int dattn_commit(dattn_t* h, int layer, const dattn_cache* cache, int num_streams, int rows, const void* k,
                 const void* v, const int32_t* parent, const int32_t* accepted, const int32_t* num_accepted,
                 const int32_t* pos, dattn_stream_t stream) {
  if (!h || layer < 0 || layer >= static_cast<int>(h->layers.size())) return DATTN_EINVAL;
  const dattn_layer_config& L = h->layers[layer];
  int rc = check_cache(L, cache);
  if (rc != DATTN_OK) return rc;
  if (num_streams <= 0 || rows <= 0 || !k || !v || !parent || !accepted || !num_accepted) return DATTN_EINVAL;
  if (L.rotary_dim > 0 && !pos) return DATTN_EINVAL;
  if (L.kv_format != DATTN_KV_BF16) return DATTN_EUNSUPPORTED;
  if (!aligned16(k) || !aligned16(v)) return DATTN_EINVAL;
  if (rows > 16) return DATTN_EXCEEDS;
  DeviceGuard guard(h->device);
  if (!guard.ok) return DATTN_ECUDA;
  // a gathered append: node accepted[b][d] to cache index start + d, rotated
  // at pos[b] + d, where start is the ring head or the prefix length
  AppendArgs a{};
  a.c = make_view(h, L, cache);
  a.B = num_streams;
  a.Tmax = rows;
  a.Hkv = h->Hkv;
  a.D = h->D;
  a.r = L.rotary_dim;
  a.start_index = L.cache_kind == DATTN_CACHE_RING ? cache->ring_head : cache->seq_len;
  a.start_pos = pos;
  a.count = num_accepted;
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.rotate = 1;
  a.rope_step = h->rope_step[layer];
  a.err = h->err;
  a.k_norm = h->k_norm[layer];
  a.norm_eps = L.norm_eps;
  a.gather = accepted;
  a.parent = parent;
  a.in_T = rows;
  rc = cuda_status(launch_append(a, reinterpret_cast<cudaStream_t>(stream)), "commit");
  if (rc == DATTN_OK) record_launch(stream, cache->k);
  return rc;
}

int dattn_decode(dattn_t* h, int layer, const dattn_cache* cache, const dattn_decode_args* args,
                 dattn_stream_t stream) {
  if (!h || !args || layer < 0 || layer >= static_cast<int>(h->layers.size())) return DATTN_EINVAL;
  const dattn_layer_config& L = h->layers[layer];
  int rc = check_cache(L, cache);
  if (rc != DATTN_OK) return rc;
  const int B = args->num_streams;
  if (B <= 0) return DATTN_EINVAL;
  if (B > h->max_streams) return DATTN_EXCEEDS;
  if (!args->q || !args->k_new || !args->v_new || !args->pos || !args->out) return DATTN_EINVAL;
  if (!aligned16(args->q) || !aligned16(args->k_new) || !aligned16(args->v_new) ||
      !aligned16(args->out))
    return DATTN_EINVAL;
  int n_max;
  if (L.cache_kind == DATTN_CACHE_RING) {
    n_max = L.ring_slots;
  } else {
    n_max = args->max_seq_len > 0 ? args->max_seq_len : h->max_context;
    if (n_max > h->max_context) return DATTN_EXCEEDS;
  }
  DeviceGuard guard(h->device);
  if (!guard.ok) return DATTN_ECUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  const bool f8 = L.kv_format == DATTN_KV_E4M3;
  const int ctas = plan_decode_ctas(h->decode_resident, B * h->Hkv, n_max, decode_tile_keys(h->D, h->G, f8));
  if (static_cast<size_t>(ctas) + static_cast<size_t>(B) * h->Hkv > h->part_units) return DATTN_EXCEEDS;
  DecodeArgs da{};
  da.c = make_view(h, L, cache);
  if (encode_cache_maps(da.c, h->Hkv, h->D, &da.tmap_k, &da.tmap_v, f8) != cudaSuccess) return DATTN_EUNSUPPORTED;
  da.B = B;
  da.Hkv = h->Hkv;
  da.G = h->G;
  da.max_len = n_max;
  da.q = static_cast<const uint16_t*>(args->q);
  da.k_new = static_cast<const uint16_t*>(args->k_new);
  da.v_new = static_cast<const uint16_t*>(args->v_new);
  da.gate = static_cast<const uint16_t*>(args->gate);
  da.pos = args->pos;
  da.rope_step = h->rope_step[layer];
  da.r = L.rotary_dim;
  da.q_scale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(h->D)));
  da.out = args->out;
  da.write_back = args->write_back;
  const unsigned half = h->decode_calls & 1u;
  da.part = h->part[half];
  da.counters = h->counters[half];
  da.err = h->err;
  da.early = !prev_launch_writes(stream, cache->k);
  da.wait_ns = h->wait_ns;
  da.debug_flags = h->debug_flags;
  da.q_norm = h->q_norm[layer];
  da.k_norm = h->k_norm[layer];
  da.norm_eps = L.norm_eps;
  if (f8) {
    // the K scale rides on q's pre-scale; V's is applied to each partial output
    da.f8 = 1;
    da.k_scale = L.k_scale;
    da.v_scale = L.v_scale;
    da.q_scale = static_cast<float>(static_cast<double>(da.q_scale) * L.k_scale);
  }
  rc = cuda_status(launch_decode(da, h->D, ctas, s), "decode");
  if (rc == DATTN_OK) {
    record_launch(stream, args->write_back ? cache->k : nullptr);
    ++h->decode_calls;
  }
  return rc;
}

int dattn_verify(dattn_t* h, int layer, const dattn_cache* cache, const dattn_verify_args* args,
                 dattn_stream_t stream) {
  if (!h || !args || layer < 0 || layer >= static_cast<int>(h->layers.size())) return DATTN_EINVAL;
  const dattn_layer_config& L = h->layers[layer];
  const bool ring = L.cache_kind == DATTN_CACHE_RING;
  // the prefix pass reads pages as 16-row groups, of bf16
  if ((!ring && L.page_size % 16 != 0) || L.kv_format != DATTN_KV_BF16) return DATTN_EUNSUPPORTED;
  int rc = check_cache(L, cache);
  if (rc != DATTN_OK) return rc;
  const int S = args->num_streams, T = args->rows;
  if (S <= 0 || T <= 0) return DATTN_EINVAL;
  if (h->max_verify_rows == 0 || T > h->max_verify_rows || S > h->max_streams) return DATTN_EXCEEDS;
  if (!args->q || !args->k || !args->v || !args->parent || !args->out) return DATTN_EINVAL;
  if (!aligned16(args->q) || !aligned16(args->k) || !aligned16(args->v) || !aligned16(args->out))
    return DATTN_EINVAL;
  // ring layers: the root positions are the caller's, and nothing is written
  if (ring && (!args->pos || args->write_back)) return DATTN_EINVAL;
  int n_max;
  if (ring) {
    n_max = L.ring_slots;
  } else {
    n_max = args->max_prefix_len > 0 ? args->max_prefix_len : h->max_context;
    if (n_max > h->max_context) return DATTN_EXCEEDS;
  }
  DeviceGuard guard(h->device);
  if (!guard.ok) return DATTN_ECUDA;
  VerifyRound vr{};
  vr.c = make_view(h, L, cache);
  vr.S = S;
  vr.T = T;
  vr.n_max = n_max;
  vr.q = static_cast<const uint16_t*>(args->q);
  vr.k = static_cast<const uint16_t*>(args->k);
  vr.v = static_cast<const uint16_t*>(args->v);
  vr.gate = static_cast<const uint16_t*>(args->gate);
  vr.parent = args->parent;
  vr.pos = args->pos ? args->pos : cache->seq_len;  // the roots' positions
  vr.out = args->out;
  vr.write_back = args->write_back;
  vr.in_T = T;
  rc = verify_round(h, layer, vr, reinterpret_cast<cudaStream_t>(stream));
  if (rc == DATTN_OK) record_launch(stream, args->write_back ? cache->k : nullptr);
  return rc;
}

int dattn_prefill(dattn_t* h, int layer, const dattn_cache* cache, int num_streams, int max_tokens,
                  const void* q, const void* k, const void* v, const void* gate, const int32_t* count,
                  const int32_t* start_pos, float* out, dattn_stream_t stream) {
  if (!h || layer < 0 || layer >= static_cast<int>(h->layers.size())) return DATTN_EINVAL;
  const dattn_layer_config& L = h->layers[layer];
  const bool ring = L.cache_kind == DATTN_CACHE_RING;
  if ((!ring && L.page_size % 16 != 0) || L.kv_format != DATTN_KV_BF16) return DATTN_EUNSUPPORTED;
  int rc = check_cache(L, cache);
  if (rc != DATTN_OK) return rc;
  const int S = num_streams;
  if (S <= 0 || max_tokens < 0 || !q || !k || !v || !count || !out) return DATTN_EINVAL;
  if (L.rotary_dim > 0 && !start_pos) return DATTN_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return DATTN_EINVAL;
  if (S > h->max_streams || h->max_verify_rows == 0) return DATTN_EXCEEDS;
  if (max_tokens == 0) return DATTN_OK;
  // chunk rows: the verify workspace's rows, at most 128 query rows per KV
  // head, and no more than a ring holds
  int Tc = std::min(h->max_verify_rows, kVerifyMaxRows / h->G);
  if (ring) Tc = std::min(Tc, L.ring_slots);
  const int n_max = ring ? L.ring_slots : h->max_context;
  DeviceGuard guard(h->device);
  if (!guard.ok) return DATTN_ECUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const CacheView base = make_view(h, L, cache);
  int32_t* seq_c = h->pmeta;
  int32_t* head_c = seq_c + h->max_streams;
  int32_t* cnt_c = head_c + h->max_streams;
  int32_t* pos_c = cnt_c + h->max_streams;
  int32_t* n_c = pos_c + h->max_streams;
  for (int row0 = 0; row0 < max_tokens; row0 += Tc) {
    // the cache as this chunk sees it: the caller's plus the earlier chunks'
    // tokens (the library never changes the caller's metadata)
    PrefillMetaArgs m{};
    m.c = base;
    m.count = count;
    m.start_pos = start_pos;
    m.S = S;
    m.Tmax = max_tokens;
    m.row0 = row0;
    m.Tc = Tc;
    m.seq_c = seq_c;
    m.head_c = head_c;
    m.cnt_c = cnt_c;
    m.pos_c = pos_c;
    m.n_c = n_c;
    m.chain = h->chain;
    m.err = h->err;
    rc = cuda_status(launch_prefill_meta(m, s), "prefill chunk state");
    if (rc != DATTN_OK) return rc;
    CacheView cv = base;
    if (ring) {
      cv.ring_head = head_c;
      cv.ring_count = cnt_c;
    } else {
      cv.seq_len = seq_c;
    }
    // the chunk's rows as chain trees through the verify pass ...
    VerifyRound vr{};
    vr.c = cv;
    vr.S = S;
    vr.T = Tc;
    vr.n_max = n_max;
    vr.q = static_cast<const uint16_t*>(q);
    vr.k = static_cast<const uint16_t*>(k);
    vr.v = static_cast<const uint16_t*>(v);
    vr.gate = static_cast<const uint16_t*>(gate);
    vr.parent = h->chain;
    vr.pos = pos_c;
    vr.out = out;
    vr.in_T = max_tokens;
    vr.row0 = row0;
    vr.rows_valid = n_c;
    vr.after_plain_launch = true;
    rc = verify_round(h, layer, vr, s);
    if (rc != DATTN_OK) return rc;
    // ... and their entries into the cache before the next chunk
    AppendArgs a{};
    a.c = cv;
    a.B = S;
    a.Tmax = Tc;
    a.Hkv = h->Hkv;
    a.D = h->D;
    a.r = L.rotary_dim;
    a.start_index = ring ? head_c : seq_c;
    a.start_pos = pos_c;
    a.count = n_c;
    a.k = static_cast<const uint16_t*>(k);
    a.v = static_cast<const uint16_t*>(v);
    a.rotate = 1;
    a.rope_step = h->rope_step[layer];
    a.err = h->err;
    a.k_norm = h->k_norm[layer];
    a.norm_eps = L.norm_eps;
    a.in_T = max_tokens;
    a.row0 = row0;
    rc = cuda_status(launch_append(a, s), "prefill commit");
    if (rc != DATTN_OK) return rc;
  }
  record_launch(stream, cache->k);
  return DATTN_OK;
}

}  // extern "C"
