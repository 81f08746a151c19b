// Microbenchmark: throughput of tcgen05.mma kind::f16 (M = 128, K = 16 per
// instruction, f32 accumulation) for the operand shapes of the tree-verify
// pass. One CTA per SM (152), one issuing thread per CTA. A "tile" is 16 MMAs
// (K = 256: the Q K^T of one 32-key tile at head_dim 256); the P V rows add
// the 2 MMAs of N = 256 that follow it. Reported: median over CTAs of the time
// per tile and per MMA.
//
// Build and run (standalone; not part of the library):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 --expt-relaxed-constexpr \
//        -I decode_attention_kv_dattn_gb300/csrc -o /tmp/tcgen05_mma_rate \
//        decode_attention_kv_dattn_gb300/microbench/tcgen05_mma_rate.cu && /tmp/tcgen05_mma_rate
//
// Every access stays inside a 192 KB shared buffer and 512 TMEM columns; the
// completion wait is bounded (an error status, never a hang).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <vector>

#include "common.cuh"
#include "tc.cuh"

using namespace dattn;

namespace {

struct Cfg {
  int a_smem;  // A from shared memory (1) or TMEM (0)
  int n;       // N of the 16 Q K^T-shaped MMAs (0: none)
  int nacc;    // k-steps spread round-robin over this many accumulators
  int accum;   // accumulate into earlier k-steps (0: every MMA overwrites)
  int pv;      // add the 2 P V MMAs (N = 256, A from TMEM) per tile
};

constexpr int kCfg = 13;
// host tables (names stay on the host), copied to the constant bank before launch
const char* const kNames[kCfg] = {
    "A tmem, N=32",          "A tmem, N=64",        "A tmem, N=128",        "A tmem, N=256",
    "A smem, N=32",          "A smem, N=128",       "A smem, N=256",        "A tmem, N=32, 2 acc",
    "A tmem, N=32, 8 acc",   "A tmem, N=32, no accum", "A tmem, N=32 + P V", "A tmem, N=64 x8 + P V",
    "P V only (2 x N=256)"};
const Cfg kHostCfgs[kCfg] = {
    {0, 32, 1, 1, 0}, {0, 64, 1, 1, 0}, {0, 128, 1, 1, 0}, {0, 256, 1, 1, 0}, {1, 32, 1, 1, 0},
    {1, 128, 1, 1, 0}, {1, 256, 1, 1, 0}, {0, 32, 2, 1, 0}, {0, 32, 8, 1, 0}, {0, 32, 1, 0, 0},
    {0, 32, 1, 1, 1}, {0, 64, 1, 1, 2}, {0, 0, 1, 1, 1}};
__constant__ Cfg cfgs[kCfg];

constexpr uint32_t kA = 0, kB = 65536, kBar = 65536 + 131072;  // shared offsets
constexpr int kSmem = kBar + 64 + 1024;

__global__ void __launch_bounds__(128, 1) mma_rate(unsigned long long* out, int reps, int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const uint32_t sA = sbase + kA, sB = sbase + kB, bar = sbase + kBar, slot = bar + 8;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < static_cast<int>(kBar / 16); i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) tc::alloc(slot, 512);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + (slot - sbase));
  {  // zero TMEM: warp w owns lanes 32w .. 32w + 31
    uint32_t z[32];
#pragma unroll
    for (int x = 0; x < 32; ++x) z[x] = 0u;
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
    for (int c = 0; c < 512; c += 32) tc::st32(tmem + lane_off + c, z);
    tc::wait_st();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  // TMEM columns: Q K^T accumulators 0..255, A (q) 256..383, P 384..399,
  // P V accumulator 256..511 (overlapping A: values are irrelevant here).
  bool ok = true;
  for (int cf = 0; cf < kCfg; ++cf) {
    const Cfg c = cfgs[cf];
    __syncthreads();
    if (threadIdx.x == 0 && ok) {
      uint32_t dcol[16];
      uint32_t accm = 0;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        dcol[kk] = static_cast<uint32_t>((kk % c.nacc) * (c.n > 0 ? c.n : 32));
        if (c.accum && kk >= c.nacc) accm |= 1u << kk;
      }
      const int nqk = c.pv == 2 ? 8 : 16;  // N=64 x8: the same keys as 16 MMAs of N=32
      const uint32_t idesc = tc::f16_idesc(128, c.n > 0 ? c.n : 32, 0, false);
      const uint32_t idesc_pv = tc::f16_idesc(128, 256, 0, true);
      const uint64_t t0 = global_timer_ns();
      for (int r = 0; r < reps; ++r) {
        if (c.n > 0) {
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            if (kk < nqk) {
              const uint64_t db = tc::sw128_desc(sB + (kk >> 2) * 32768 + (kk & 3) * 32, 16, 1024);
              const bool acc = (accm >> kk) & 1u;
              if (c.a_smem) {
                const uint64_t da = tc::sw128_desc(sA + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                tc::mma(tmem + dcol[kk], da, db, idesc, acc);
              } else {
                tc::mma_ts(tmem + dcol[kk], tmem + 256 + kk * 8, db, idesc, acc);
              }
            }
          }
        }
        if (c.pv) {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            tc::mma_ts(tmem + 256, tmem + 384 + kk * 8, tc::sw128_desc(sB + kk * 2048, 4096, 1024), idesc_pv,
                       true);
        }
      }
      tc::commit(bar);
      ok = mbar_wait_bounded(bar, cf & 1);
      const uint64_t t1 = global_timer_ns();
      if (!ok) atomicExch(status, 1);
      out[blockIdx.x * kCfg + cf] = t1 - t0;
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::dealloc(tmem, 512);
  }
}

}  // namespace

int main() {
  const int ctas = 152, reps = 256;
  unsigned long long* d_out = nullptr;
  int* d_status = nullptr;
  cudaMalloc(&d_out, ctas * kCfg * sizeof(unsigned long long));
  cudaMalloc(&d_status, sizeof(int));
  cudaMemset(d_status, 0, sizeof(int));
  cudaMemcpyToSymbol(cfgs, kHostCfgs, sizeof(kHostCfgs));
  cudaFuncSetAttribute(mma_rate, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  for (int it = 0; it < 3; ++it) mma_rate<<<ctas, 128, kSmem>>>(d_out, reps, d_status);
  const cudaError_t e = cudaDeviceSynchronize();
  std::vector<unsigned long long> h(ctas * kCfg);
  int st = 0;
  cudaMemcpy(h.data(), d_out, h.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  cudaMemcpy(&st, d_status, sizeof(int), cudaMemcpyDeviceToHost);
  printf("kernel: %s, status %d (%d CTAs, one per SM, %d tiles each)\n", cudaGetErrorString(e), st, ctas, reps);
  for (int cf = 0; cf < kCfg; ++cf) {
    std::vector<double> t;
    for (int b = 0; b < ctas; ++b) t.push_back(h[b * kCfg + cf] / static_cast<double>(reps));
    std::sort(t.begin(), t.end());
    const Cfg& c = kHostCfgs[cf];
    const int nmma = (c.n > 0 ? (c.pv == 2 ? 8 : 16) : 0) + (c.pv ? 2 : 0);
    printf("%-24s %2d MMAs per tile: %7.1f ns per tile, %5.1f ns per MMA\n", kNames[cf], nmma, t[ctas / 2],
           t[ctas / 2] / nmma);
  }
  cudaFree(d_out);
  cudaFree(d_status);
  return e == cudaSuccess && st == 0 ? 0 : 1;
}
