/*
 * dattn: decode attention over per-stream KV caches on one GB300 (sm_103a).
 *
 * One query token per stream attends to that stream's cached keys and values
 * plus its own new key and value. Two cache layouts are supported:
 *
 *   ring  - a sliding-window layer keeps window-1 slots per (stream, KV head);
 *           the valid slots are the `count` slots before `head` (cyclically),
 *           in any order. ("vllm-omni commits", score-space join commit: the
 *           ring needs no reordering because softmax is order-free and each
 *           cached key already carries its rotary phase; only unwritten slots
 *           are masked; a 512-token window holds 511 cached entries.)
 *   paged - a full-attention layer keeps its tokens in fixed-size pages named
 *           by a per-stream page table ("pega-omni PR #4": talker KV in paged
 *           leases; padding rows of a call name a pad page).
 *
 * The new token is joined in score space: the cache and the new key are
 * scored separately and the two score vectors meet in one softmax, so nothing
 * cache-sized is copied; the call returns the new K/V entry by writing it into
 * its slot (same commit). RoPE is applied per layer type to the new q and k
 * ("vllm-omni commits", Spark model commit: sliding layers rotate all 256 dims
 * with theta 1e4, full layers the first quarter with theta 5e6), and an
 * optional head-wise sigmoid gate scales each head's output (same commit).
 * Grouped-query attention maps query head h to KV head h / (Hq / Hkv)
 * ("vllm-omni commits", talker export commit: GQA by reshaping the query).
 * Tree verify scores up to 16 rows per stream, each under its own tree mask
 * ("TensorFold PR #608": verify windows of up to 16 streams x 16 rows).
 *
 * Conventions for every entry point:
 *   - All tensor and index pointers are DEVICE pointers on the handle's GPU,
 *     owned by the caller, dense row-major in the layouts stated below. bf16
 *     data is passed as raw 16-bit patterns. Pointers must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream); the
 *     calls that take a handle may be captured in a CUDA graph. Calls that
 *     share one handle use its workspace and must be ordered (one stream, or
 *     one handle per stream).
 *   - The return value is a dattn status. Host-side argument checks return
 *     DATTN_EINVAL / DATTN_EXCEEDS / DATTN_EUNSUPPORTED before anything is
 *     launched. Bad device-side metadata (a page id outside the pool, a ring
 *     head outside [0, R), a length above the planned bound, a bad tree parent)
 *     never faults: the kernel skips or clamps the access and sets a sticky
 *     device error word that dattn_get_error() reports.
 *   - The library never mutates caller metadata: after a call the caller
 *     advances ring head/count or seq_len itself.
 */
#ifndef DATTN_H
#define DATTN_H

#include <stddef.h>
#include <stdint.h>

#ifndef DATTN_API
#define DATTN_API __attribute__((visibility("default")))
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum {
  DATTN_OK = 0,
  DATTN_EINVAL = 1,        /* invalid argument (null pointer, bad shape)         */
  DATTN_EXCEEDS = 2,       /* beyond what dattn_create planned for (cf. the
                              pages' ExceedsPool: rejected, not queued forever)  */
  DATTN_ECUDA = 3,         /* a CUDA runtime call failed                          */
  DATTN_EINDEX = 4,        /* device metadata out of range (from dattn_get_error) */
  DATTN_ETIMEOUT = 5,      /* a bounded device wait gave up (dattn_get_error)     */
  DATTN_EUNSUPPORTED = 6,  /* a shape with no compiled kernel                     */
  DATTN_ELENGTH = 7,       /* a stream longer than the call's bound (get_error)   */
  DATTN_ERANGE = 8         /* verify: a cached V value beyond the fp16 range
                              (|x| >= 65520) in which the tensor-core pass forms
                              P V (from dattn_get_error)                          */
};

enum { DATTN_CACHE_RING = 0, DATTN_CACHE_PAGED = 1 };

/* Element format of a layer's K/V pools. */
enum {
  DATTN_KV_BF16 = 0,  /* bf16 (raw 16-bit patterns)                                 */
  DATTN_KV_E4M3 = 1   /* OCP FP8 E4M3 bytes; value = e4m3 * scale ("TensorFold PR
                         #608" names the fp8 cache and leaves it out): decode and
                         append only                                              */
};

/* cudaStream_t without including the CUDA headers. */
typedef struct CUstream_st* dattn_stream_t;

/* Per-layer description, copied by dattn_create. */
typedef struct {
  int cache_kind;     /* DATTN_CACHE_RING or DATTN_CACHE_PAGED                   */
  int ring_slots;     /* ring: R = window - 1 slots per (row, KV head)           */
  int page_size;      /* paged: P tokens per page (P * head_dim * 2 % 16 == 0)   */
  int rotary_dim;     /* r: RoPE turns dims [0, r) in pairs (i, i + r/2); even,
                         <= head_dim; 0 = no rotation                            */
  double rope_theta;  /* base of the inverse frequencies theta^(-2i/r)           */
  /* QK-norm before RoPE ("pega-omni PR #4", talker kernels: RoPE with QK-norm),
   * per head: y_d = w_d x_d / sqrt(mean(x^2) + eps), rounded once to bf16 (ties
   * to even), then RoPE turns y. HOST pointers to [head_dim] bf16 weights,
   * copied by dattn_create (dattn_decode_noalloc copies them on each call);
   * NULL = no norm for that side. The key side applies to the new token of
   * decode, the window rows of verify and dattn_append_kv with rotate != 0. */
  const uint16_t* q_norm_weight;
  const uint16_t* k_norm_weight;
  double norm_eps;    /* eps (>= 0) of both norms                               */
  /* DATTN_KV_BF16 (0) or DATTN_KV_E4M3. An E4M3 layer's pools hold bytes
   * [.., D] instead of bf16; a cached K value is e4m3 * k_scale, a V value
   * e4m3 * v_scale (finite, > 0; quantisation divides by these fp32 values
   * in fp64). Decode scores the cache as stored, stores
   * the new entry as the E4M3 bytes nearest entry / k_scale and
   * v_new / v_scale (ties to even, saturating at 448) and joins the new token
   * as stored; dattn_append_kv stores the same bytes. dattn_verify,
   * dattn_commit, dattn_prefill and dattn_decode_noalloc return
   * DATTN_EUNSUPPORTED for such a layer. */
  int kv_format;
  float k_scale;
  float v_scale;
} dattn_layer_config;

typedef struct {
  int num_q_heads;       /* Hq                                                   */
  int num_kv_heads;      /* Hkv; Hq % Hkv == 0                                   */
  int head_dim;          /* D: 128 or 256                                         */
  int max_streams;       /* largest B of a decode call / S of a verify call       */
  int max_context;       /* largest cached length of a paged stream; calls with a
                            longer bound return DATTN_EXCEEDS                      */
  int max_verify_rows;   /* largest T of a verify call (<= 16); 0 = no verify     */
  int num_layers;
  const dattn_layer_config* layers; /* [num_layers], host memory                  */
} dattn_config;

typedef struct dattn_handle dattn_t;

/* One layer's cache as the caller holds it. Ring fields are read for ring
 * layers, paged fields for paged layers.
 *   ring : k, v = [n_rows, Hkv, R, D] bf16. Call row b uses ring row
 *          stream_rows[b] (identity when NULL); its valid slots are the
 *          ring_count[b] slots before ring_head[b]; the new entry is written
 *          at slot ring_head[b].
 *   paged: k, v = [n_rows (pages), Hkv, P, D] bf16. Token t of call row b is
 *          offset t % P of page block_table[b * bt_stride + t / P]; the row
 *          holds seq_len[b] cached tokens; the new entry is written at token
 *          index seq_len[b]. */
typedef struct {
  void* k;
  void* v;
  int n_rows;
  const int32_t* ring_head;    /* [B] */
  const int32_t* ring_count;   /* [B] */
  const int32_t* stream_rows;  /* [B] or NULL */
  const int32_t* block_table;  /* [B, bt_stride] */
  int bt_stride;
  const int32_t* seq_len;      /* [B] */
} dattn_cache;

/* One decode step: B streams, one new token each. */
typedef struct {
  int num_streams;       /* B, 1 <= B <= max_streams                             */
  const void* q;         /* [B, Hq, D] bf16                                       */
  const void* k_new;     /* [B, Hkv, D] bf16, before RoPE                         */
  const void* v_new;     /* [B, Hkv, D] bf16                                      */
  const void* gate;      /* [B, Hq] bf16 gate logits, or NULL for no gate        */
  const int32_t* pos;    /* [B] RoPE position of the new token                    */
  float* out;            /* [B, Hq, D] fp32: sigmoid(gate) * attention output     */
  int max_seq_len;       /* paged: host-side bound on seq_len[b] for this call
                            (0 = max_context); sizes the key split. Ignored for
                            ring layers (the bound is R).                          */
  int write_back;        /* nonzero: store the rotated bf16 k_new and v_new into
                            the new token's slot after every read of the cache   */
} dattn_decode_args;

/* One verify round: S streams x T rows ("TensorFold PR #608": verify windows
 * under tree masks). Row i of stream s sits at position pos[s] + depth(i)
 * (depth 0 for a root); it attends to its ancestors in the tree, to itself -
 * each window key rotated at its own position - and to the stream's cache:
 *   paged layer: the whole prefix of seq_len[s] tokens;
 *   ring layer : the newest min(ring_count[s], R - depth(i)) entries of its
 *                ring, what the ring holds once the row's ancestors have been
 *                appended (a verify row equals the plain decode of its path).
 * Ring layers are never written by verify: dattn_commit writes the accepted
 * path. */
typedef struct {
  int num_streams;       /* S                                                     */
  int rows;              /* T, 1 <= T <= max_verify_rows                          */
  const void* q;         /* [S, T, Hq, D] bf16                                    */
  const void* k;         /* [S, T, Hkv, D] bf16, before RoPE                      */
  const void* v;         /* [S, T, Hkv, D] bf16                                   */
  const int32_t* parent; /* [S, T]: parent[i] < i, or -1 for a root              */
  const void* gate;      /* [S, T, Hq] bf16 or NULL                               */
  float* out;            /* [S, T, Hq, D] fp32                                    */
  int max_prefix_len;    /* host bound on seq_len[s] (0 = max_context)            */
  int write_back;        /* paged layers: nonzero writes window entry i to token
                            index seq_len[s] + i (node order). Ring layers: must
                            be 0 (DATTN_EINVAL otherwise)                         */
  const int32_t* pos;    /* [S] position of the window's root, or NULL for
                            seq_len[s] (paged layers only: ring layers need it)   */
} dattn_verify_args;

/* Create a handle on `device`: validates the config, uploads per-layer RoPE
 * phase-step tables (the angle per position of each pair, theta^(-2i/r), as
 * 64-bit fixed-point turns, computed on the host) and
 * allocates the workspace: the split-K partials and per-(stream, KV head)
 * segment counters of decode, and the verify pass's buffers. The handle owns
 * that memory until dattn_destroy. */
DATTN_API int dattn_create(const dattn_config* cfg, int device, dattn_t** out);

/* Bulk write (prefill or cache set-up): token t < count[b] of call row b goes
 * to cache index start_index[b] + t (ring: slot (start_index[b] + t) mod R of
 * row stream_rows[b]; paged: offset idx % P of page block_table[b][idx / P]).
 * k, v = [B, max_tokens, Hkv, D] bf16. A ring row takes at most R tokens per
 * call (count[b] > R is reported as DATTN_EINDEX and writes nothing for b). When rotate != 0 the key is turned at
 * position start_pos[b] + t and rounded to the bf16 nearest the exact
 * rotation (ties to even) - the same entry decode writes back. start_index, start_pos, count: [B]. */
DATTN_API int dattn_append_kv(dattn_t* h, int layer, const dattn_cache* cache, int num_streams,
                    int max_tokens, const int32_t* start_index, const int32_t* start_pos,
                    const int32_t* count, const void* k, const void* v, int rotate,
                    dattn_stream_t stream);

/* Decode attention for one layer (see dattn_decode_args). One kernel launch.
 * Ordering: calls on one handle share its workspace, so they must be ordered
 * (one stream at a time, or streams joined by events). The launch may begin
 * while the launch before it on the stream is still running: it then streams
 * its cache early, but only when that earlier launch (a decode, verify or
 * append of this library) does not write into the same cache; its outputs and
 * the write-back always wait for the earlier launch to complete. Inputs (q,
 * k_new, v_new, gate, pos, cache metadata) must not be produced by the
 * immediately preceding launch if that launch is one of this library's. */
DATTN_API int dattn_decode(dattn_t* h, int layer, const dattn_cache* cache, const dattn_decode_args* args,
                 dattn_stream_t stream);

/* Tree verify for one layer, ring or paged (see dattn_verify_args). Three
 * launches. Shape limits: G * T <= 128 query rows per KV head and
 * num_streams * Hkv <= 512 (checked at dattn_create: DATTN_EUNSUPPORTED); a
 * paged layer's page size is a multiple of 16. */
DATTN_API int dattn_verify(dattn_t* h, int layer, const dattn_cache* cache, const dattn_verify_args* args,
                 dattn_stream_t stream);

/* Commit of a verify round ("TensorFold PR #608": a round commits only each
 * stream's accepted path). accepted [S, T] lists stream s's accepted nodes
 * root first, num_accepted[s] (0..T) of them; they must form a path from a
 * root (accepted[0] has parent -1, each next node is a child of the one
 * before). Node accepted[s][d] is written at cache index start + d - ring:
 * slot (ring_head[s] + d) mod R of ring row stream_rows[s]; paged: token index
 * seq_len[s] + d - with its key normalised (QK-norm) and rotated at
 * pos[s] + d: the same bf16 entry that verify scored for that node and that
 * a decode of the path would write. k, v, parent: the verify call's window
 * inputs [S, T, Hkv, D] and [S, T]; pos [S]: the root positions. A stream
 * whose list is not such a path writes nothing and is reported as
 * DATTN_EINDEX (dattn_get_error). The caller then advances ring head/count
 * or seq_len by num_accepted[s]. One launch. */
DATTN_API int dattn_commit(dattn_t* h, int layer, const dattn_cache* cache, int num_streams, int rows,
                           const void* k, const void* v, const int32_t* parent, const int32_t* accepted,
                           const int32_t* num_accepted, const int32_t* pos, dattn_stream_t stream);

/* Ragged prefill ("TensorFold PR #608" and "pega-omni PR #4": prefill rows
 * beside the decode steps): stream s brings count[s] (0..max_tokens) new
 * tokens, token t at position start_pos[s] + t. Each token attends to the
 * stream's cache and to new tokens 0..t, and every new entry is written to
 * the cache (ring: slot head + t, the ring keeping its newest R entries;
 * paged: token index seq_len[s] + t) - the same as decoding the tokens one
 * after another with write-back. q [S, max_tokens, Hq, D], k, v [S, max_tokens,
 * Hkv, D] bf16, gate [S, max_tokens, Hq] or NULL; out [S, max_tokens, Hq, D]
 * fp32: rows t < count[s] are written, the others are left as they are.
 * The tokens go through the verify pass in chunks of min(max_verify_rows,
 * 128 / G, R) rows as chain trees, each chunk committed before the next
 * (five launches per chunk), so the handle needs max_verify_rows > 0
 * (DATTN_EXCEEDS otherwise); a paged stream's cache must hold its new tokens
 * (seq_len[s] + count[s] <= max_context, pages in its table). A stream whose
 * count or ring metadata is out of range gets no tokens and is reported as
 * DATTN_EINDEX (dattn_get_error). The caller then advances its metadata by
 * count[s]. */
DATTN_API int dattn_prefill(dattn_t* h, int layer, const dattn_cache* cache, int num_streams, int max_tokens,
                            const void* q, const void* k, const void* v, const void* gate,
                            const int32_t* count, const int32_t* start_pos, float* out, dattn_stream_t stream);

/* Synchronize `stream`, then return and clear the sticky device error word:
 * DATTN_OK, DATTN_ETIMEOUT, DATTN_EINDEX, DATTN_ERANGE or DATTN_ELENGTH (the
 * first found in that order of severity). */
DATTN_API int dattn_get_error(dattn_t* h, dattn_stream_t stream);

/* Testing aid for the failure path (no counterpart on the pages): every
 * device wait of the library is bounded, and one that runs out ends the call
 * with DATTN_ETIMEOUT from dattn_get_error instead of hanging the GPU.
 *   wait_limit_us - limit of the handle's bounded waits in microseconds for
 *                   its later decode calls (0 = the default, 2 s).
 *   flags         - DATTN_DEBUG_WITHHOLD_Q: in each later decode call, the
 *                   kernel's helper warp withholds every CTA's first rotated
 *                   query, so the streaming warps' waits for it run out after
 *                   the limit. The call still completes (the copies it issued
 *                   land before it exits) and the context stays usable; the
 *                   output and any write-back of that call are undefined.
 *                   0 restores normal operation.
 * Returns DATTN_EINVAL for a null handle or an unknown flag. */
enum { DATTN_DEBUG_WITHHOLD_Q = 1 };
DATTN_API int dattn_debug_config(dattn_t* h, int flags, unsigned wait_limit_us);

/* Static description of a status code. */
DATTN_API const char* dattn_error_string(int code);

/* Free the workspace and the handle. Safe on NULL. */
DATTN_API void dattn_destroy(dattn_t* h);

/* Decode for callers that cannot allocate device memory (no counterpart on the
 * pages: it serves callers whose device memory is owned by someone else, e.g.
 * a server that hands out its whole pool up front, or code that must not
 * allocate inside a latency-critical loop). Same operation, layouts and
 * arguments as dattn_decode for layer `layer` of `cfg`, but no handle: the
 * scratch space (split partials, per-unit segment counters, error word, RoPE
 * phase steps) lives in one 8 MiB array in device memory that the library
 * defines at file scope; every GPU that loads the library holds it until the
 * process exits. Nothing is allocated or freed by this call.
 *   - The first call on a device looks up the array's device address (with
 *     that device current).
 *   - A call whose scratch would not fit in 8 MiB returns DATTN_EXCEEDS
 *     (about 1.2 MiB for 64 streams x 2 KV heads x 8 query heads x head_dim
 *     256 on a 152-SM GPU).
 *   - All calls on a device share the array, which keeps the last call's
 *     contents. Each call first runs a small set-up kernel that clears the
 *     error word and the segment counters and writes the RoPE phase steps
 *     (passed by value), then the decode kernel; calls that overlap on the
 *     GPU (other streams, or unordered) race on the array.
 *   - Device-side metadata errors (a page id outside the pool, a ring head
 *     outside [0, R), a length above the bound) are recorded in the array's
 *     error word and are not returned; only host-side checks produce the
 *     status. The output of a call with such metadata is undefined. */
DATTN_API int dattn_decode_noalloc(const dattn_config* cfg, int layer, const dattn_cache* cache,
                                   const dattn_decode_args* args, dattn_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DATTN_H */
