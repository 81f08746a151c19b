// dattn_decode_noalloc: decode attention for callers that cannot allocate
// device memory.
//
// Some callers have no way to call cudaMalloc: code that runs inside a memory
// budget owned by someone else (an inference server that hands out all device
// memory from its own pool up front), code that must not allocate while a
// latency-critical loop runs, or embedding layers that only receive raw device
// pointers. dattn_create allocates the handle's workspace, so those callers
// cannot use dattn_decode. This entry point needs no handle: its scratch space
// (the split partials, the per-unit segment counters, the error word and the
// RoPE phase-step table and the layer's QK-norm weights) lives in one fixed-size array in device global memory
// that the library defines at file scope. The caller passes only its inputs,
// outputs and cache, exactly as for dattn_decode.
//
// The array is created when the library's module is loaded on a device and
// stays there until the process exits. All calls on a device share it and it
// keeps the last call's contents. Every call starts with a small set-up kernel
// that clears the error word and the segment counters (the decode kernel
// needs them at zero) and writes the layer's RoPE phase steps and QK-norm
// weights, which it receives by value in its kernel parameters - no host buffer has to outlive
// the call. Two calls that run on the GPU at the same time - on different
// streams, or not ordered on one stream - race on the array.
//
// The decode kernel is the same one dattn_decode launches; only where its
// scratch lives differs, and it is launched as an ordinary (not a
// programmatic-dependent) launch, so it starts after the set-up kernel has
// completed.
#include <cmath>
#include <mutex>

#include "dattn.h"
#include "kernels.h"

using namespace dattn;

namespace {

// Upper bound of the scratch this entry point may use on one device: 8 MiB.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct DeviceScratch {
  bool ready = false;
  unsigned char* base = nullptr;  // device address of g_noalloc_scratch
  int sms = 0;
};

constexpr int kMaxDevices = 64;
DeviceScratch g_devices[kMaxDevices];
std::mutex g_mutex;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

constexpr int kMaxPhaseSteps = 128;  // r / 2 for r <= 256
constexpr int kMaxHeadDim = 256;

// Everything the set-up kernel writes, passed by value.
struct NoAllocSetup {
  uint64_t step[kMaxPhaseSteps];  // RoPE phase steps of the layer
  uint64_t* step_dst;
  uint16_t norm[2][kMaxHeadDim];  // QK-norm weights (queries, keys)
  uint16_t* norm_dst[2];          // or null for a side without a norm
  int D;
  int half;                       // r / 2
  int* err;
  int* counters;
  int n_counters;
};

__global__ void __launch_bounds__(256) noalloc_setup_kernel(const __grid_constant__ NoAllocSetup p) {
  for (int i = threadIdx.x; i < p.half; i += blockDim.x) p.step_dst[i] = p.step[i];
  for (int side = 0; side < 2; ++side)
    if (p.norm_dst[side])
      for (int i = threadIdx.x; i < p.D; i += blockDim.x) p.norm_dst[side][i] = p.norm[side][i];
  for (int i = threadIdx.x; i < p.n_counters; i += blockDim.x) p.counters[i] = 0;
  if (threadIdx.x == 0) *p.err = 0;
}

}  // namespace

extern "C" DATTN_API int dattn_decode_noalloc(const dattn_config* cfg, int layer, const dattn_cache* cache,
                                              const dattn_decode_args* args, dattn_stream_t stream) {
  // ---- host checks (nothing is launched when one fails)
  if (!cfg || !cache || !args || !cfg->layers || layer < 0 || layer >= cfg->num_layers) return DATTN_EINVAL;
  const int Hq = cfg->num_q_heads, Hkv = cfg->num_kv_heads, D = cfg->head_dim;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return DATTN_EINVAL;
  if (D != 128 && D != 256) return DATTN_EUNSUPPORTED;
  const int G = Hq / Hkv, GP = decode_group_pad(G);
  if (GP == 0) return DATTN_EUNSUPPORTED;
  const dattn_layer_config& L = cfg->layers[layer];
  if (L.rotary_dim < 0 || L.rotary_dim > D || L.rotary_dim % 2 || (L.rotary_dim > 0 && !(L.rope_theta > 0.0)))
    return DATTN_EINVAL;
  if ((L.q_norm_weight || L.k_norm_weight) && !(L.norm_eps >= 0.0)) return DATTN_EINVAL;
  if (L.kv_format != DATTN_KV_BF16) return DATTN_EUNSUPPORTED;
  if (!cache->k || !cache->v || cache->n_rows <= 0) return DATTN_EINVAL;
  if ((reinterpret_cast<uintptr_t>(cache->k) | reinterpret_cast<uintptr_t>(cache->v)) & 15u) return DATTN_EINVAL;
  int n_max;
  if (L.cache_kind == DATTN_CACHE_RING) {
    if (L.ring_slots <= 0 || !cache->ring_head || !cache->ring_count) return DATTN_EINVAL;
    n_max = L.ring_slots;
  } else if (L.cache_kind == DATTN_CACHE_PAGED) {
    if (L.page_size <= 0 || !cache->block_table || !cache->seq_len || cache->bt_stride <= 0) return DATTN_EINVAL;
    n_max = args->max_seq_len > 0 ? args->max_seq_len : cfg->max_context;
    if (n_max <= 0 || n_max > cfg->max_context) return DATTN_EXCEEDS;
  } else {
    return DATTN_EINVAL;
  }
  const int B = args->num_streams;
  if (B <= 0) return DATTN_EINVAL;
  if (!args->q || !args->k_new || !args->v_new || !args->pos || !args->out) return DATTN_EINVAL;
  if ((reinterpret_cast<uintptr_t>(args->q) | reinterpret_cast<uintptr_t>(args->k_new) |
       reinterpret_cast<uintptr_t>(args->v_new) | reinterpret_cast<uintptr_t>(args->out)) & 15u)
    return DATTN_EINVAL;
  if (static_cast<int64_t>(B) * Hkv > decode_max_units()) return DATTN_EXCEEDS;

  // ---- once per device: the device address of the scratch array
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DATTN_ECUDA;
  DeviceScratch ds;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceScratch& d = g_devices[dev];
    if (!d.ready) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return DATTN_ECUDA;
      int sms = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DATTN_ECUDA;
      d.base = static_cast<unsigned char*>(p);
      d.sms = sms;
      d.ready = true;
    }
    ds = d;
  }

  // ---- the grid, as dattn_decode plans it
  const int tile_keys = decode_tile_keys(D, G);
  const int resident = ds.sms * decode_ctas_per_sm(D, G);
  if (tile_keys <= 0 || resident <= 0) return DATTN_EUNSUPPORTED;
  const int ctas = plan_decode_ctas(resident, B * Hkv, n_max, tile_keys);

  // ---- carve the scratch; reject what does not fit
  const int half = L.rotary_dim / 2;
  if (half > kMaxPhaseSteps) return DATTN_EUNSUPPORTED;
  size_t off = 0;
  const size_t err_off = off;
  off = align256(off + sizeof(int));
  const size_t freq_off = off;
  off = align256(off + static_cast<size_t>(half) * sizeof(uint64_t));
  const size_t norm_off = off;
  off = align256(off + 2 * static_cast<size_t>(D) * sizeof(uint16_t));
  const size_t counters_off = off;
  off = align256(off + (static_cast<size_t>(B) * Hkv + ctas) * sizeof(int));  // units, then one per CTA
  const size_t part_off = off;
  off = align256(off + (static_cast<size_t>(ctas) + static_cast<size_t>(B) * Hkv) * GP * (D + 2) * sizeof(float));
  if (off > kNoAllocScratchBytes) return DATTN_EXCEEDS;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* err = reinterpret_cast<int*>(ds.base + err_off);
  CacheView cv{};
  cv.k = static_cast<uint16_t*>(cache->k);
  cv.v = static_cast<uint16_t*>(cache->v);
  cv.paged = L.cache_kind == DATTN_CACHE_PAGED;
  cv.n_rows = cache->n_rows;
  cv.R = L.ring_slots;
  cv.P = L.page_size;
  cv.ring_head = cache->ring_head;
  cv.ring_count = cache->ring_count;
  cv.stream_rows = cache->stream_rows;
  cv.block_table = cache->block_table;
  cv.bt_stride = cache->bt_stride;
  cv.seq_len = cache->seq_len;
  // the kernel reads the cache through tensor maps (host-side encoding)
  DecodeArgs da{};
  if (encode_cache_maps(cv, Hkv, D, &da.tmap_k, &da.tmap_v) != cudaSuccess) return DATTN_EUNSUPPORTED;

  uint64_t* rope_step = half > 0 ? reinterpret_cast<uint64_t*>(ds.base + freq_off) : nullptr;
  int* counters = reinterpret_cast<int*>(ds.base + counters_off);
  // The error word accumulates bits and the segment counters must start at
  // zero, so both are cleared every call, and the RoPE phase steps are
  // rewritten, by one set-up kernel that holds the steps in its parameters.
  NoAllocSetup setup{};
  for (int i = 0; i < half; ++i) setup.step[i] = rope_phase_step(L.rope_theta, L.rotary_dim, i);
  setup.step_dst = rope_step;
  uint16_t* norm_dev[2] = {nullptr, nullptr};
  for (int side = 0; side < 2; ++side) {
    const uint16_t* w = side == 0 ? L.q_norm_weight : L.k_norm_weight;
    if (!w) continue;
    for (int i = 0; i < D; ++i) setup.norm[side][i] = w[i];
    norm_dev[side] = reinterpret_cast<uint16_t*>(ds.base + norm_off) + side * D;
    setup.norm_dst[side] = norm_dev[side];
  }
  setup.D = D;
  setup.half = half;
  setup.err = err;
  setup.counters = counters;
  setup.n_counters = B * Hkv + ctas;
  noalloc_setup_kernel<<<1, 256, 0, s>>>(setup);
  if (cudaGetLastError() != cudaSuccess) return DATTN_ECUDA;

  da.c = cv;
  da.B = B;
  da.Hkv = Hkv;
  da.G = G;
  da.max_len = n_max;
  da.q = static_cast<const uint16_t*>(args->q);
  da.k_new = static_cast<const uint16_t*>(args->k_new);
  da.v_new = static_cast<const uint16_t*>(args->v_new);
  da.gate = static_cast<const uint16_t*>(args->gate);
  da.pos = args->pos;
  da.rope_step = rope_step;
  da.r = L.rotary_dim;
  da.q_scale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  da.out = args->out;
  da.write_back = args->write_back;
  da.part = reinterpret_cast<float*>(ds.base + part_off);
  da.counters = counters;
  da.err = err;
  da.early = !prev_launch_writes(stream, cache->k);
  da.q_norm = norm_dev[0];
  da.k_norm = norm_dev[1];
  da.norm_eps = L.norm_eps;
  const cudaError_t e = launch_decode(da, D, ctas, s, /*pdl=*/false);
  if (e != cudaSuccess) return e == cudaErrorNotSupported ? DATTN_EUNSUPPORTED : DATTN_ECUDA;
  record_launch(stream, args->write_back ? cache->k : nullptr);
  return DATTN_OK;
}
