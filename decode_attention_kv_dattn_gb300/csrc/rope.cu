// RoPE prologue of a decode or verify call, and the bulk append kernel.
//
// Per-layer-type RoPE ("vllm-omni commits", Spark model commit): sliding
// layers turn all 256 head dims with theta 1e4, full layers the first quarter
// with theta 5e6. Pair i of the first r dims is (i, i + r/2) and turns by
// pos * theta^(-2i/r) (rotate-half convention); dims >= r pass through.
//
// Rounding contract of the K entry (the value stored in the cache and scored
// for the new token): angle = pos * inv_freq in fp64, with inv_freq computed on
// the host in fp64; c and s are the fp64 cosine and sine rounded to fp32; the
// entry is bf16_RNE(x*c - y*s) evaluated in fp64. Each product of a bf16 and an
// fp32 value is exact in fp64, so the only roundings are the fp64 difference
// and the final bf16 step. q is rotated in fp32 and pre-scaled by
// log2(e)/sqrt(D) so that the split kernel's scores are in base-2 units.
#include "common.cuh"

namespace dattn {

namespace {

constexpr int kRopeThreads = 64;

// Position of verify row `row` = s*T + i: prefix_len[s] + depth(i), walking
// the parent pointers (parent[i] < i, -1 = root). A bad parent stops the walk
// and is reported.
__device__ __forceinline__ int64_t verify_position(const RopeArgs& a, int row, int* err) {
  const int s = row / a.T;
  const int i = row - s * a.T;
  const int32_t* par = a.parent + static_cast<int64_t>(s) * a.T;
  int depth = 0;
  int node = i;
  for (int steps = 0; steps < a.T; ++steps) {
    const int p = par[node];
    if (p < 0) break;
    if (p >= node) {
      raise_error(err, ERR_INDEX);
      break;
    }
    ++depth;
    node = p;
  }
  return static_cast<int64_t>(a.prefix_len[s]) + depth;
}

__global__ void __launch_bounds__(kRopeThreads) rope_kernel(const RopeArgs a) {
  // The workspace written below may still be read by the previous call.
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y;
  const int job = blockIdx.x * kRopeThreads + threadIdx.x;
  const int half = a.r / 2;
  if (job >= half + (a.D - a.r)) return;
  const int64_t pos = a.parent ? verify_position(a, row, a.err) : a.pos[row];
  const uint16_t* q = a.q + static_cast<int64_t>(row) * a.Hq * a.D;
  const uint16_t* k = a.k + static_cast<int64_t>(row) * a.Hkv * a.D;
  float* qh = a.qhat + static_cast<int64_t>(row) * a.Hq * a.D;
  uint16_t* kh = a.khat + static_cast<int64_t>(row) * a.Hkv * a.D;
  if (job < half) {
    const int i = job;
    const double angle = __dmul_rn(static_cast<double>(pos), a.inv_freq[i]);
    double sd, cd;
    sincos(angle, &sd, &cd);
    const float cf = __double2float_rn(cd);
    const float sf = __double2float_rn(sd);
    for (int h = 0; h < a.Hq; ++h) {
      const float x = bf16_to_f32(q[h * a.D + i]);
      const float y = bf16_to_f32(q[h * a.D + i + half]);
      qh[h * a.D + i] = fmaf(x, cf, -y * sf) * a.q_scale;
      qh[h * a.D + i + half] = fmaf(y, cf, x * sf) * a.q_scale;
    }
    const double c64 = cf, s64 = sf;
    for (int h = 0; h < a.Hkv; ++h) {
      const double x = bf16_to_f32(k[h * a.D + i]);
      const double y = bf16_to_f32(k[h * a.D + i + half]);
      kh[h * a.D + i] = f64_to_bf16(__dsub_rn(__dmul_rn(x, c64), __dmul_rn(y, s64)));
      kh[h * a.D + i + half] = f64_to_bf16(__dadd_rn(__dmul_rn(y, c64), __dmul_rn(x, s64)));
    }
  } else {
    const int d = a.r + (job - half);
    for (int h = 0; h < a.Hq; ++h) qh[h * a.D + d] = bf16_to_f32(q[h * a.D + d]) * a.q_scale;
    for (int h = 0; h < a.Hkv; ++h) kh[h * a.D + d] = k[h * a.D + d];
  }
}

// One CTA per (token t, call row b): writes the token's K/V rows of every KV
// head into its ring slot or page slot.
__global__ void __launch_bounds__(kRopeThreads) append_kernel(const AppendArgs a) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x, b = blockIdx.y;
  const CacheView& c = a.c;
  const int cnt = a.count[b];
  if (cnt < 0 || cnt > a.Tmax) {
    if (t == 0 && threadIdx.x == 0) raise_error(a.err, ERR_INDEX);
    return;
  }
  if (t >= cnt) return;
  const int64_t idx = static_cast<int64_t>(a.start_index[b]) + t;
  if (idx < 0) {
    if (threadIdx.x == 0) raise_error(a.err, ERR_INDEX);
    return;
  }
  // Destination row base for KV head 0; heads are D * rows_per_head apart.
  int64_t dst0;
  int64_t head_stride;
  if (c.paged) {
    const int64_t pi = idx / c.P;
    const int pg = pi < c.bt_stride ? c.block_table[static_cast<int64_t>(b) * c.bt_stride + pi] : -1;
    if (pg < 0 || pg >= c.n_rows) {
      if (threadIdx.x == 0) raise_error(a.err, ERR_INDEX);
      return;
    }
    dst0 = (static_cast<int64_t>(pg) * a.Hkv * c.P + idx % c.P) * a.D;
    head_stride = static_cast<int64_t>(c.P) * a.D;
  } else {
    const int row = c.stream_rows ? c.stream_rows[b] : b;
    if (row < 0 || row >= c.n_rows) {
      if (threadIdx.x == 0) raise_error(a.err, ERR_INDEX);
      return;
    }
    dst0 = (static_cast<int64_t>(row) * a.Hkv * c.R + idx % c.R) * a.D;
    head_stride = static_cast<int64_t>(c.R) * a.D;
  }
  const int64_t src0 = (static_cast<int64_t>(b) * a.Tmax + t) * a.Hkv * a.D;
  // V: plain copy, 16 bytes per thread-step.
  for (int e = threadIdx.x; e < a.Hkv * a.D / 8; e += kRopeThreads) {
    const int h = e / (a.D / 8), d8 = e % (a.D / 8);
    const uint4 w = *reinterpret_cast<const uint4*>(a.v + src0 + h * a.D + d8 * 8);
    *reinterpret_cast<uint4*>(c.v + dst0 + h * head_stride + d8 * 8) = w;
  }
  if (!a.rotate || a.r == 0) {
    for (int e = threadIdx.x; e < a.Hkv * a.D / 8; e += kRopeThreads) {
      const int h = e / (a.D / 8), d8 = e % (a.D / 8);
      const uint4 w = *reinterpret_cast<const uint4*>(a.k + src0 + h * a.D + d8 * 8);
      *reinterpret_cast<uint4*>(c.k + dst0 + h * head_stride + d8 * 8) = w;
    }
    return;
  }
  const int half = a.r / 2;
  const int64_t pos = static_cast<int64_t>(a.start_pos[b]) + t;
  for (int job = threadIdx.x; job < half + (a.D - a.r); job += kRopeThreads) {
    if (job < half) {
      const int i = job;
      const double angle = __dmul_rn(static_cast<double>(pos), a.inv_freq[i]);
      double sd, cd;
      sincos(angle, &sd, &cd);
      const double c64 = __double2float_rn(cd), s64 = __double2float_rn(sd);
      for (int h = 0; h < a.Hkv; ++h) {
        const double x = bf16_to_f32(a.k[src0 + h * a.D + i]);
        const double y = bf16_to_f32(a.k[src0 + h * a.D + i + half]);
        c.k[dst0 + h * head_stride + i] =
            f64_to_bf16(__dsub_rn(__dmul_rn(x, c64), __dmul_rn(y, s64)));
        c.k[dst0 + h * head_stride + i + half] =
            f64_to_bf16(__dadd_rn(__dmul_rn(y, c64), __dmul_rn(x, s64)));
      }
    } else {
      const int d = a.r + (job - half);
      for (int h = 0; h < a.Hkv; ++h) c.k[dst0 + h * head_stride + d] = a.k[src0 + h * a.D + d];
    }
  }
}

}  // namespace

cudaError_t launch_rope(const RopeArgs& a, cudaStream_t s) {
  const int jobs = a.r / 2 + (a.D - a.r);
  dim3 grid((jobs + kRopeThreads - 1) / kRopeThreads, a.rows);
  return launch_pdl(rope_kernel, grid, dim3(kRopeThreads), 0, s, a);
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
  dim3 grid(a.Tmax, a.B);
  return launch_pdl(append_kernel, grid, dim3(kRopeThreads), 0, s, a);
}

}  // namespace dattn
