// Tensor-core rate probe, a measurement aid for the roofline of the fused
// kernels: the dense kind::f16 rate of one SM, measured rather than taken
// from a data sheet.
//
// Each CTA (one per SM: its shared-memory request leaves room for no second
// CTA) holds one 128 x 64 A slice (K-major) and one 64 x 256 B slice
// (N-major, four 64-column boxes), both 128-byte swizzled exactly as the
// fused kernels stage their operands, and zero-filled.  One thread issues
// `iters` x 4 back-to-back tcgen05.mma.cta_group::1.kind::f16 of M = 128,
// N = 256, K = 16 into one TMEM accumulator -- no loads, no epilogue -- then
// a commit, and records the SM clock cycles and %globaltimer nanoseconds
// from the first issue to the commit's arrival.  FLOP per MMA =
// 2 * 128 * 256 * 16, so FLOP per SM clock = iters * 4 * 2^20 / cycles, and
// the clock the probe ran at = cycles / ns.  The wait is bounded (about 4 s);
// a wait that runs out is reported in the CTA's record.
#include "tc_ptx.cuh"

namespace bra {
namespace {

using namespace tc;

constexpr int kProbeThreads = 128;
constexpr int kProbeA = 128 * 64 * 2;     // A slice bytes
constexpr int kProbeB = 64 * 256 * 2;     // B slice bytes (four 8 KiB boxes)
// Shared memory requested per CTA: above half of an SM's, so CTAs never share one.
constexpr int kProbeSmem = 160 * 1024;
constexpr uint32_t kProbeCols = 256;

__device__ int32_t g_probe_fault_word = 0;

__global__ void __launch_bounds__(kProbeThreads, 1)
    mma_probe_kernel(int iters, uint32_t idesc, int64_t* rec) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5;

  uint4* z = reinterpret_cast<uint4*>(smem);
  for (int k = tid; k < (kProbeA + kProbeB) / 16; k += kProbeThreads) z[k] = make_uint4(0, 0, 0, 0);
  // The operands were written by ordinary stores; the tensor core reads them
  // through the async proxy.
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(&tmem_slot), kProbeCols);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (tid == 0) {
    const uint32_t a = smem_u32(smem), b = a + kProbeA;
    const uint64_t ad = smem_desc_sw128(a, 16, 1024);
    const uint64_t bd = smem_desc_sw128(b, 8192, 1024);
    const long long c0 = clock64();
    const unsigned long long g0 = global_ns();
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int k = 0; k < 4; ++k) tc_mma<1>(tmem, ad + 2 * k, bd + 128 * k, idesc, 1u);
    }
    tc_commit(smem_u32(&bar));
    const bool ok = mbar_wait(smem_u32(&bar), 0, &abort_flag, &g_probe_fault_word);
    const long long c1 = clock64();
    const unsigned long long g1 = global_ns();
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    int64_t* r = rec + 4 * (int64_t)blockIdx.x;
    r[0] = c1 - c0;
    r[1] = (int64_t)(g1 - g0);
    r[2] = ok ? BRA_OK : BRA_ERR_TIMEOUT;
    r[3] = smid;
    if (!ok) spin_ns(2000000ull);   // MMAs already issued complete
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<1>(tmem, kProbeCols);
  }
}

}  // namespace

cudaError_t launch_mma_probe(int ctas, int iters, bool bf16, int64_t* rec, cudaStream_t st) {
  static std::mutex mu;
  static bool ready[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!ready[dev & 63]) {
      e = cudaFuncSetAttribute(mma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kProbeSmem);
      if (e != cudaSuccess) return e;
      ready[dev & 63] = true;
    }
  }
  mma_probe_kernel<<<ctas, kProbeThreads, kProbeSmem, st>>>(iters, make_idesc(bf16, 128, 256),
                                                            rec);
  return cudaGetLastError();
}

}  // namespace bra
