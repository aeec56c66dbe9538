// all_to_all_v among P virtual ranks resident on one GPU.
//
// Semantics ("LowerL2TensorCollectives Pass", 行为 / ABI; addressing as in
// the meta ncclx alltoallv of "vccl alltoallv dev log", 5. ref): rank i sends
// send_counts[i][j] elements to rank j; displacements are exclusive prefix
// sums in element units, over destinations for the sender and over sources
// for the receiver.
//
// One launch, grid (ctas_per_rank, P), sized to fill the GPU about once.
// Every CTA of source rank i:
//   1. stages the whole P x P count matrix in shared memory (P <= 64, rows
//      padded to P+1 so column reads hit distinct banks) and rejects the call
//      if any count is negative or a NULL buffer would be touched (every CTA
//      sees the same matrix, so all take the same decision without a grid
//      sync);
//   2. warp-scans row i (its send displacements) and, per column j, the
//      counts of sources k < i (its receive displacement at rank j);
//   3. CTA 0 of rank i writes row i of send_displs and column i of
//      recv_counts / recv_displs;
//   4. copies: rank i's send buffer is split into B = CalAllToAllVBlocks(P, L)
//      equal element ranges ("blocks"); each CTA takes a contiguous run of
//      blocks and cuts it at the destination boundaries into at most P
//      pieces.  Head and tail bytes of a piece (before its first / after its
//      last 16-byte-aligned destination vector) are copied byte by byte; the
//      vector part is cut into tiles of up to kTileVecs vectors.  One thread
//      streams the tiles' source words into a kStages-deep shared-memory ring
//      with cp.async.bulk (TMA bulk copies, completion on an mbarrier);
//      seven consumer warps shift each tile's words into destination
//      alignment (int8 can be off by any byte, fp32 by whole words) and write
//      16-byte vectors.  Up to kStages tiles per CTA are in flight without
//      holding registers.
// Every wait is bounded (about 2 s by %globaltimer); a wait that runs out
// records BRA_ERR_TIMEOUT in this file's device word, flags the CTA, and all
// roles leave their loops.
#include <cstdint>
#include <mutex>

#include "bra_internal.h"

namespace bra {

__device__ int32_t g_a2av_fault_word = 0;

namespace {

constexpr unsigned kFull = 0xffffffffu;
#ifndef BRA_A2AV_STAGES
#define BRA_A2AV_STAGES 4
#endif
#ifndef BRA_A2AV_TILE_VECS
#define BRA_A2AV_TILE_VECS 1024
#endif
#ifndef BRA_A2AV_MIN_CTAS
#define BRA_A2AV_MIN_CTAS 2
#endif
constexpr int kStages = BRA_A2AV_STAGES;
constexpr int kTileVecs = BRA_A2AV_TILE_VECS;            // 16-byte destination vectors
constexpr int kStageBytes = (kTileVecs + 1) * 16;        // + one word when shifted
constexpr int kStageStride = (kStageBytes + 127) / 128 * 128;
constexpr int kRingBytes = kStages * kStageStride;
constexpr int kConsumerWarps = kA2avThreads / 32 - 1;
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

// Exclusive scan of 64 values held as (lane, lane + 32) by one warp.
__device__ __forceinline__ void warp_exscan64(int64_t v0, int64_t v1, int lane,
                                              int64_t& ex0, int64_t& ex1,
                                              int64_t& total) {
  int64_t s0 = v0, s1 = v1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t n0 = __shfl_up_sync(kFull, s0, o);
    const int64_t n1 = __shfl_up_sync(kFull, s1, o);
    if (lane >= o) {
      s0 += n0;
      s1 += n1;
    }
  }
  const int64_t t0 = __shfl_sync(kFull, s0, 31);
  const int64_t t1 = __shfl_sync(kFull, s1, 31);
  ex0 = s0 - v0;
  ex1 = t0 + s1 - v1;
  total = t0 + t1;
}

// The 16 destination bytes that start `delta` bytes into the 32 source bytes
// (a, b), which start at an aligned address: shift by whole words (q =
// delta / 4, in two select stages), then by the remaining bytes (r = 8 *
// (delta % 4) bits) with funnel shifts.  One code path for every delta.
__device__ __forceinline__ uint4 realign(const uint4& a, const uint4& b, uint32_t q, uint32_t r) {
  const bool two = (q & 2u) != 0, one = (q & 1u) != 0;
  const uint32_t x0 = two ? a.z : a.x, x1 = two ? a.w : a.y, x2 = two ? b.x : a.z;
  const uint32_t x3 = two ? b.y : a.w, x4 = two ? b.z : b.x, x5 = two ? b.w : b.y;
  const uint32_t y0 = one ? x1 : x0, y1 = one ? x2 : x1, y2 = one ? x3 : x2;
  const uint32_t y3 = one ? x4 : x3, y4 = one ? x5 : x4;
  uint4 o;
  o.x = __funnelshift_r(y0, y1, r);
  o.y = __funnelshift_r(y1, y2, r);
  o.z = __funnelshift_r(y2, y3, r);
  o.w = __funnelshift_r(y3, y4, r);
  return o;
}

// Start of equal range b of B over n elements (ranges differ by at most one).
__device__ __forceinline__ int64_t split_point(int64_t n, int64_t B, int64_t b) {
  const int64_t q = n / B, rem = n % B;
  return q * b + (b < rem ? b : rem);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
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
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int k = 0; k < 64; ++k)
      if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitTimeoutNs) {
      *abort_flag = 1;
      atomicExch(&g_a2av_fault_word, (int32_t)BRA_ERR_TIMEOUT);
      return false;
    }
  }
}
// Bulk copy of `bytes` (a multiple of 16) from a 16-byte-aligned global
// address into shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__global__ void __launch_bounds__(kA2avThreads, BRA_A2AV_MIN_CTAS)
a2av_kernel(const __grid_constant__ A2avArgs a) {
  extern __shared__ __align__(128) uint8_t ring[];   // kStages x kStageStride
  __shared__ int64_t s_sc[kA2avMaxP * (kA2avMaxP + 1)];   // row stride P + 1
  __shared__ int64_t s_sd[kA2avMaxP];    // send displacement of rank i to j
  __shared__ int64_t s_rd[kA2avMaxP];    // receive displacement of i at j
  __shared__ int64_t s_tot[kA2avMaxP];   // elements rank j receives
  // This CTA's share of rank i's send buffer, cut at destination
  // boundaries: one piece per destination j (possibly empty).
  __shared__ const char* s_src[kA2avMaxP];   // first source byte of the piece
  __shared__ char* s_dst[kA2avMaxP];         // first destination byte
  __shared__ int64_t s_nvec[kA2avMaxP];      // 16-byte destination vectors
  __shared__ int s_head[kA2avMaxP];          // bytes before the first vector
  __shared__ int s_tail[kA2avMaxP];          // bytes after the last vector
  __shared__ int64_t s_tile0[kA2avMaxP + 1]; // first tile of each piece
  __shared__ __align__(8) uint64_t s_full[kStages];
  __shared__ __align__(8) uint64_t s_empty[kStages];
  __shared__ int s_bad;
  __shared__ int s_abort;

  const int P = a.P;
  const int i = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;

  if (tid == 0) {
    s_bad = 0;
    s_abort = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&s_full[s]), 1);
      mbar_init(smem_u32(&s_empty[s]), kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int ld = P + 1;   // padded row stride: column reads hit distinct banks
  for (int k = tid; k < P * P; k += blockDim.x) {
    const int64_t v = a.sc[k];
    s_sc[(k / P) * ld + k % P] = v;
    if (v < 0) s_bad = 1;
  }
  __syncthreads();

  // Bookkeeping: warp-scanned prefix sums of row i and of every column.
  if (warp == 0) {
    const int64_t v0 = lane < P ? s_sc[i * ld + lane] : 0;
    const int64_t v1 = lane + 32 < P ? s_sc[i * ld + lane + 32] : 0;
    int64_t e0, e1, tot;
    warp_exscan64(v0, v1, lane, e0, e1, tot);
    if (lane < P) s_sd[lane] = e0;
    if (lane + 32 < P) s_sd[lane + 32] = e1;
  }
  for (int j = warp; j < P; j += nwarps) {
    const int64_t v0 = lane < P ? s_sc[lane * ld + j] : 0;
    const int64_t v1 = lane + 32 < P ? s_sc[(lane + 32) * ld + j] : 0;
    int64_t e0, e1, tot;
    warp_exscan64(v0, v1, lane, e0, e1, tot);
    const int64_t at_i = __shfl_sync(kFull, i < 32 ? e0 : e1, i & 31);
    if (lane == 0) {
      s_rd[j] = at_i;
      s_tot[j] = tot;
    }
  }
  __syncthreads();

  // Data checks every CTA takes identically: a NULL buffer that would be
  // read or written, and (checked variant) a receive total over capacity.
  if (tid < P && !s_bad) {
    int64_t row = 0;
    for (int k = 0; k < P; ++k) row += s_sc[tid * ld + k];
    if (a.in[tid] == nullptr && row > 0) s_bad = 1;
    if (a.out[tid] == nullptr && s_tot[tid] > 0) s_bad = 1;
    if (a.check_cap && s_tot[tid] > a.cap[tid]) s_bad = 1;
  }
  __syncthreads();
  const bool bad = s_bad != 0;
  if (a.status && blockIdx.x == 0 && i == 0 && tid == 0)
    *a.status = bad ? BRA_ERR_INVALID : BRA_OK;
  if (bad) return;

  if (blockIdx.x == 0) {
    for (int j = tid; j < P; j += blockDim.x) {
      a.sd[(int64_t)i * P + j] = s_sd[j];
      a.rc[(int64_t)j * P + i] = s_sc[i * ld + j];
      a.rd[(int64_t)j * P + i] = s_rd[j];
    }
  }

  // This CTA's contiguous range: logical blocks [b0, b1) of the B equal
  // ranges rank i's send buffer is split into.
  const int64_t total = s_sd[P - 1] + s_sc[i * ld + P - 1];
  const int64_t b0 = (int64_t)blockIdx.x * a.B / gridDim.x;
  const int64_t b1 = (int64_t)(blockIdx.x + 1) * a.B / gridDim.x;
  const int64_t lo = split_point(total, a.B, b0), hi = split_point(total, a.B, b1);
  const int64_t es = a.esize;

  if (warp == 0) {
    int64_t ntile[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = lane + 32 * h;
      ntile[h] = 0;
      if (j < P) {
        const int64_t seg_lo = s_sd[j], seg_hi = seg_lo + s_sc[i * ld + j];
        const int64_t c0 = lo > seg_lo ? lo : seg_lo;
        const int64_t c1 = hi < seg_hi ? hi : seg_hi;
        const int64_t n = c1 > c0 ? (c1 - c0) * es : 0;
        const char* src = static_cast<const char*>(a.in[i]) + (n ? c0 * es : 0);
        char* dst = static_cast<char*>(a.out[j]) + (n ? (s_rd[j] + (c0 - seg_lo)) * es : 0);
        int64_t head = (16 - (int64_t)((uintptr_t)dst & 15)) & 15;
        if (head > n) head = n;
        const int64_t nvec = (n - head) >> 4;
        s_src[j] = src;
        s_dst[j] = dst;
        s_head[j] = (int)head;
        s_nvec[j] = nvec;
        s_tail[j] = (int)((n - head) & 15);
        ntile[h] = (nvec + kTileVecs - 1) / kTileVecs;
      }
    }
    int64_t e0, e1, tot;
    warp_exscan64(ntile[0], ntile[1], lane, e0, e1, tot);
    if (lane < P) s_tile0[lane] = e0;
    if (lane + 32 < P) s_tile0[lane + 32] = e1;
    if (lane == 0) s_tile0[P] = tot;
  }
  __syncthreads();

  // Vector parts: a bulk-copy producer and kConsumerWarps consumer warps.
  const int64_t ntiles = s_tile0[P];
  volatile int* abort_flag = &s_abort;
  const uint32_t ring_base = smem_u32(ring);
  if (warp == 0) {
    if (lane == 0) {
      int j = 0, stage = 0;
      uint32_t phase = 0;
      bool ok = true;
#pragma unroll 1
      for (int64_t t = 0; t < ntiles; ++t) {
        while (s_tile0[j + 1] <= t) ++j;
        if (!mbar_wait(smem_u32(&s_empty[stage]), phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const int64_t v0 = (t - s_tile0[j]) * kTileVecs;
        const int64_t left = s_nvec[j] - v0;
        const int n = left < kTileVecs ? (int)left : kTileVecs;
        const char* src = s_src[j] + s_head[j] + v0 * 16;
        const uint32_t delta = (uint32_t)((uintptr_t)src & 15);
        const uint32_t bytes = (uint32_t)(n + (delta ? 1 : 0)) * 16u;
        const uint32_t fb = smem_u32(&s_full[stage]);
        mbar_expect_tx(fb, bytes);
        bulk_load(ring_base + stage * kStageStride, src - delta, bytes, fb);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {   // let copies already issued land before the CTA exits
        const unsigned long long t0 = global_ns();
        while (global_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else {
    const int ctid = tid - 32, nct = kConsumerWarps * 32;
    // Head and tail bytes of every piece, while the first tiles are in flight.
#pragma unroll 1
    for (int k = ctid; k < P * 32; k += nct) {
      const int jj = k >> 5, b = k & 31;
      if (b < 16) {
        if (b < s_head[jj]) s_dst[jj][b] = s_src[jj][b];
      } else if (b - 16 < s_tail[jj]) {
        const int64_t off = s_head[jj] + s_nvec[jj] * 16 + (b - 16);
        s_dst[jj][off] = s_src[jj][off];
      }
    }
    int j = 0, stage = 0;
    uint32_t phase = 0;
#pragma unroll 1
    for (int64_t t = 0; t < ntiles; ++t) {
      while (s_tile0[j + 1] <= t) ++j;
      const bool waited = mbar_wait(smem_u32(&s_full[stage]), phase, abort_flag);
      if (!__all_sync(kFull, waited)) break;
      const int64_t v0 = (t - s_tile0[j]) * kTileVecs;
      const int64_t left = s_nvec[j] - v0;
      const int n = left < kTileVecs ? (int)left : kTileVecs;
      const char* src = s_src[j] + s_head[j] + v0 * 16;
      const uint32_t delta = (uint32_t)((uintptr_t)src & 15);
      uint4* d4 = reinterpret_cast<uint4*>(s_dst[j] + s_head[j]) + v0;
      const uint32_t buf = ring_base + stage * kStageStride;
      if (delta == 0) {
        for (int k = ctid; k < n; k += nct) d4[k] = lds128(buf + 16u * k);
      } else {
        const uint32_t q = delta >> 2, r = (delta & 3u) * 8u;
        for (int k = ctid; k < n; k += nct)
          d4[k] = realign(lds128(buf + 16u * k), lds128(buf + 16u * k + 16u), q, r);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_empty[stage]));
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n > 0 ? n : 148;
}

// Per device: the dynamic shared-memory opt-in and the resident CTA count.
struct A2avDeviceInfo {
  bool ready = false;
  int resident = 0;
};

cudaError_t a2av_device_setup(int* resident) {
  static std::mutex mu;
  static A2avDeviceInfo info[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  A2avDeviceInfo& di = info[dev & 63];
  if (!di.ready) {
    e = cudaFuncSetAttribute(a2av_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, a2av_kernel, kA2avThreads,
                                                      kRingBytes);
    if (e != cudaSuccess) return e;
    di.resident = (per_sm > 0 ? per_sm : 1) * device_sm_count();
    di.ready = true;
  }
  *resident = di.resident;
  return cudaSuccess;
}

}  // namespace

int a2av_ctas_per_rank(int P, int B) {
  int resident = 0;
  if (a2av_device_setup(&resident) != cudaSuccess || resident < 1) resident = device_sm_count();
  // Whole waves only: round down, at least one CTA per rank, at most B.
  long long c = resident / P;
  if (c < 1) c = 1;
  if (c > B) c = B;
  return (int)c;
}

cudaError_t launch_a2av(const A2avArgs& a, int ctas_per_rank, cudaStream_t st) {
  int resident = 0;
  cudaError_t e = a2av_device_setup(&resident);
  if (e != cudaSuccess) return e;
  dim3 grid(ctas_per_rank, a.P);
  a2av_kernel<<<grid, kA2avThreads, kRingBytes, st>>>(a);
  return cudaGetLastError();
}

cudaError_t read_a2av_fault_word(int32_t* code, int clear) {
  cudaError_t e = cudaMemcpyFromSymbol(code, g_a2av_fault_word, sizeof(int32_t));
  if (e != cudaSuccess) return e;
  if (clear) {
    const int32_t z = 0;
    e = cudaMemcpyToSymbol(g_a2av_fault_word, &z, sizeof(int32_t));
  }
  return e;
}

}  // namespace bra
