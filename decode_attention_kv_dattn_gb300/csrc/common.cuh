// Device helpers shared by the dattn kernels: bf16 unpacking, exp2, mbarrier
// and bulk-copy (TMA) PTX, programmatic dependent launch, bounded waits and
// the sticky error word.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "rope_angle.h"

namespace dattn {

// ------------------------------------------------------------------ numbers

// bf16 pair packed in a 32-bit word: the element at the lower address is the
// low half. Widening bf16 to fp32 is a shift (or a mask) of the bit pattern.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// fp32 -> bf16, round to nearest even (finite inputs; NaN stays NaN).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0;
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// ------------------------------------------------------------------ RoPE angle
// rope_cos_sin: rope_angle.h (plain C++ apart from the qualifiers, so that the
// host test suite builds the same routine).

// 2^x with the hardware approximation (MUFU.EX2); exact 0 for -inf.
__device__ __forceinline__ float exp2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ errors

__device__ __forceinline__ void raise_error(int* err, int bits) {
  if (err) atomicOr(err, bits);
}

// ------------------------------------------------------------------ shared memory, mbarrier, bulk copy

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Non-blocking test of phase `parity` (for polling several barriers at once:
// try_wait may suspend the thread while another barrier is already complete).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of an mbarrier, giving up after `limit_ns`
// nanoseconds (then the caller records DATTN_ETIMEOUT and leaves).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// L2 policy for data read once (the KV stream).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Contiguous global -> shared copy by the TMA unit; completion is counted on
// the mbarrier as transaction bytes. dst, src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ programmatic dependent launch

// Wait until the preceding grid in the stream has completed and its memory is
// visible (a no-op when the kernel was not launched as a dependent).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next grid in the stream to begin launching.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ loads

// Bring the 128-byte line holding p into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Inclusive prefix sum of x[0, n) in shared memory by a whole block of NT
// threads (NT a multiple of 32, at most 1024).
template <int NT>
__device__ void block_scan_inclusive(int* x, int n) {
  __shared__ int warp_sum[NT / 32];
  const int t = threadIdx.x;
  const int per = (n + NT - 1) / NT;
  const int lo = min(n, t * per), hi = min(n, lo + per);
  int sum = 0;
  for (int i = lo; i < hi; ++i) {
    sum += x[i];
    x[i] = sum;
  }
  int incl = sum;
#pragma unroll
  for (int w = 1; w < 32; w <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, w);
    if ((t & 31) >= w) incl += y;
  }
  if ((t & 31) == 31) warp_sum[t >> 5] = incl;
  __syncthreads();
  int before = incl - sum;
  for (int w = 0; w < (t >> 5); ++w) before += warp_sum[w];
  for (int i = lo; i < hi; ++i) x[i] += before;
  __syncthreads();
}

// Last unit u in [0, U) with P[u] <= g (P[0] = 0 <= g); its tile range
// [P[u], P[u + 1]) then contains g.
__host__ __device__ __forceinline__ int unit_of(const int* P, int U, int g) {
  int lo = 0, hi = U - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P[mid] <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ------------------------------------------------------------------ stream-K split

// The stream-K split runs over weighted positions: unit u starts at
// P[u] + C u, its first C positions stand for the fixed cost of one segment of
// it (what a CTA does once for every unit it takes part in: inputs, partial
// state, output), and its tiles follow one position each. CTA c takes the positions
// [c W / NC, (c + 1) W / NC) of the W = T + C U in all, so a CTA whose range
// crosses many short units gets fewer tiles.
struct Split {
  const int* P;  // [U + 1] tile prefix over units
  int U, C, NC;
  int64_t W;
  __host__ __device__ __forceinline__ int64_t bound(int c) const { return static_cast<int64_t>(c) * W / NC; }
  // first tile at or after weighted position t (T past the end)
  __host__ __device__ __forceinline__ int tile_at(int64_t t) const {
    if (t >= W) return P[U];
    int lo = 0, hi = U - 1;  // the last unit starting at or before t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (P[mid] + static_cast<int64_t>(C) * mid <= t) lo = mid; else hi = mid - 1;
    }
    const int64_t off = t - (P[lo] + static_cast<int64_t>(C) * lo) - C;
    return P[lo] + (off > 0 ? static_cast<int>(off) : 0);
  }
  // CTA whose range holds tile x of unit u
  __host__ __device__ __forceinline__ int cta_of(int x, int u) const {
    const int64_t w = x + static_cast<int64_t>(C) * (u + 1);
    return static_cast<int>(((w + 1) * NC - 1) / W);
  }
  __host__ __device__ __forceinline__ bool has_tiles_inside(int c) const { return bound(c) < bound(c + 1); }
};

// Number of CTAs whose ranges hold tiles of unit u (global tiles [p0, p1)),
// the first of them, the last, and the partial slot of the first one's
// segment (that CTA's own slot when the unit starts its range).
__host__ __device__ __forceinline__ int unit_segments(const Split& sp, int p0, int p1, int u, int& c_lo, int& c_hi,
                                             int& first_slot) {
  if (p1 <= p0) return 0;
  c_lo = sp.cta_of(p0, u);
  c_hi = sp.cta_of(p1 - 1, u);
  first_slot = sp.tile_at(sp.bound(c_lo)) == p0 ? c_lo : sp.NC + u;
  int n = 1;
  // a CTA strictly inside the unit's span holds its tiles iff its range is not empty
  for (int cc = c_lo + 1; cc <= c_hi; ++cc) n += sp.has_tiles_inside(cc);
  return n;
}

}  // namespace dattn
