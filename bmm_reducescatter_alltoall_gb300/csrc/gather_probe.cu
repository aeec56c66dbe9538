// Gather-rate probe, a measurement aid for the indexed exchange's roofline:
// how many random one-byte loads an SM completes per clock when each load
// falls in its own 128-byte line, measured rather than assumed.  The indexed
// exchange gathers its payload through a permutation, so every element it
// moves costs one such load; its bound is this rate, not HBM bandwidth.
//
// Each CTA (1024 threads; its shared-memory request leaves room for no
// second CTA on the SM) runs `iters` rounds.  In a round every thread issues
// eight independent one-byte loads at pseudo-random offsets of `buf` (a
// counter-based integer hash of the thread and load, masked to the buffer's
// power-of-two size) and then adds them up, so the loads cannot be dropped.
// Thread 0 records the SM clock cycles and %globaltimer nanoseconds of the
// loop, the SM id and the CTA's byte sum.  There is no wait: the loop ends by
// itself.
#include <mutex>

#include "bra_internal.h"

namespace bra {
namespace {

constexpr int kGatherThreads = 1024;
constexpr int kGatherUnroll = 8;
constexpr int kGatherSmem = 120 * 1024;   // above half of an SM's: one CTA per SM

__device__ __forceinline__ uint32_t hash32(uint32_t x) {
  // integer finaliser: xor-shift / multiply rounds (C. Wellons' "lowbias32")
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

__global__ void __launch_bounds__(kGatherThreads, 1)
    gather_probe_kernel(const uint8_t* __restrict__ buf, uint64_t mask, int iters, int64_t* rec) {
  extern __shared__ uint8_t unused_smem[];
  (void)unused_smem;
  __shared__ unsigned long long block_sum;
  if (threadIdx.x == 0) block_sum = 0;
  __syncthreads();
  uint32_t s = hash32(blockIdx.x * kGatherThreads + threadIdx.x + 1u);
  uint32_t acc = 0;
  long long c0 = 0;
  unsigned long long g0 = 0;
  if (threadIdx.x == 0) {
    c0 = clock64();
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(g0));
  }
#pragma unroll 1
  for (int i = 0; i < iters; ++i) {
    uint32_t v[kGatherUnroll];
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      s = hash32(s + (uint32_t)u);
      const uint64_t off = (((uint64_t)s << 16) ^ (uint64_t)hash32(s ^ 0x9e3779b9u)) & mask;
      v[u] = __ldg(buf + off);
    }
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) acc += v[u];
  }
  atomicAdd(&block_sum, (unsigned long long)acc);
  __syncthreads();
  if (threadIdx.x == 0) {
    const long long c1 = clock64();
    unsigned long long g1;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(g1));
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    int64_t* r = rec + 4 * (int64_t)blockIdx.x;
    r[0] = c1 - c0;
    r[1] = (int64_t)(g1 - g0);
    r[2] = smid;
    r[3] = (int64_t)block_sum;
  }
}

}  // namespace

cudaError_t launch_gather_probe(const void* buf, int64_t bytes, int ctas, int iters, int64_t* rec,
                                cudaStream_t st) {
  static std::mutex mu;
  static bool ready[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!ready[dev & 63]) {
      e = cudaFuncSetAttribute(gather_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kGatherSmem);
      if (e != cudaSuccess) return e;
      ready[dev & 63] = true;
    }
  }
  gather_probe_kernel<<<ctas, kGatherThreads, kGatherSmem, st>>>(
      static_cast<const uint8_t*>(buf), (uint64_t)bytes - 1, iters, rec);
  return cudaGetLastError();
}

}  // namespace bra
