// all_to_all_v among P virtual ranks resident on one GPU.
//
// Semantics ("LowerL2TensorCollectives Pass", 行为 / ABI; addressing as in
// the meta ncclx alltoallv of "vccl alltoallv dev log", 5. ref): rank i sends
// send_counts[i][j] elements to rank j; displacements are exclusive prefix
// sums in element units, over destinations for the sender and over sources
// for the receiver.
//
// One launch, grid (ctas_per_rank, P), sized to fill the GPU once whatever
// the launch width B = CalAllToAllVBlocks(P, L): B is the number of vector
// cores an Ascend launch uses, which has no counterpart here, and the results
// do not depend on how the copy is spread over CTAs.
// Every CTA of source rank i:
//   1. stages the whole P x P count matrix in shared memory (P <= 64, rows
//      padded to P+1 so column reads hit distinct banks) and rejects the call
//      if any count is negative, a non-zero count would touch a NULL buffer
//      or (checked variant) a receive total is over capacity (every CTA sees
//      the same matrix, so all take the same decision without a grid sync);
//   2. warp-scans row i (its send displacements) and sums, per column j, the
//      counts of sources k < i (its receive displacement at rank j) and of
//      all sources (what rank j receives);
//   3. CTA 0 of rank i writes row i of send_displs and column i of
//      recv_counts / recv_displs;
//   4. copies: rank i's send buffer is split into one equal element range
//      per CTA, cut at the destination boundaries into at most P pieces; a
//      piece is its 16-byte-aligned destination vectors plus head and tail
//      bytes before the first / after the last vector.  The CTA's source
//      bytes are contiguous, so one thread streams them through a
//      kStages-deep shared-memory ring in chunks of kChunk bytes (16-byte
//      granules, each chunk staged with one granule of overlap) with
//      cp.async.bulk (TMA bulk copies, completion on an mbarrier).  For each
//      chunk, seven consumer warps write every vector of every piece whose
//      first source byte lies in the chunk, shifting the words into
//      destination alignment (int8 can be off by any byte, fp32 by whole
//      words), and 32 lanes write the head and tail bytes that lie in it.  A
//      granule holding a byte of the buffer never crosses a page the buffer
//      does not touch, so the granule-wide loads stay in bounds.  Up to
//      kStages chunks per CTA are in flight without holding registers.
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
// Source bytes a chunk writes out; it is staged with one granule more.
constexpr uint32_t kChunk = kTileVecs * 16;
constexpr int kStageBytes = kChunk + 16;
constexpr int kStageStride = (kStageBytes + 127) / 128 * 128;
constexpr int kRingBytes = kStages * kStageStride;
static_assert(kRingBytes >= kA2avMaxP * (kA2avMaxP + 1) * 8, "the ring also holds the counts");
constexpr int kConsumerWarps = kA2avThreads / 32 - 1;
// The warp that scans this CTA's own row of counts.
constexpr int kRowWarp = kA2avThreads / 32 - 1;
#ifndef BRA_A2AV_PREFETCH_KB
#define BRA_A2AV_PREFETCH_KB 256
#endif
// Bytes of a CTA's source range prefetched into L2 during the set-up.
constexpr uint32_t kPrefetchBytes = BRA_A2AV_PREFETCH_KB * 1024u;
// Count-matrix entries (P x P) per thread.
constexpr int kCountIters = kA2avMaxP * kA2avMaxP / kA2avThreads;
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

// The 16 destination bytes that start Q words + r bits into the 32 source
// bytes (a, b), which start at an aligned address: word Q + k of the pair
// funnel-shifted with word Q + k + 1.  Q is fixed per instantiation, so the
// word choice costs nothing; r = 8 * (byte offset % 4) is uniform per tile.
template <int Q>
__device__ __forceinline__ uint4 realign(const uint4& a, const uint4& b, uint32_t r) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint4 o;
  o.x = __funnelshift_r(w[Q], w[Q + 1], r);
  o.y = __funnelshift_r(w[Q + 1], w[Q + 2], r);
  o.z = __funnelshift_r(w[Q + 2], w[Q + 3], r);
  o.w = __funnelshift_r(w[Q + 3], w[Q + 4], r);
  return o;
}

// Start of equal range b of B over n elements (ranges differ by at most one).
// 32-bit division whenever n fits, which every buffer below 4 G elements does.
__device__ __forceinline__ int64_t split_point(int64_t n, uint32_t B, uint32_t b) {
  if ((uint64_t)n <= 0xffffffffull) {
    const uint32_t q = (uint32_t)n / B, rem = (uint32_t)n - q * B;
    return (int64_t)q * b + (b < rem ? b : rem);
  }
  const int64_t q = n / (int64_t)B, rem = n - q * (int64_t)B;
  return q * (int64_t)b + ((int64_t)b < rem ? (int64_t)b : rem);
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
// Hint: bring `bytes` (a multiple of 16) from a 16-byte-aligned global
// address into L2.
__device__ __forceinline__ void l2_prefetch(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
               ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Copy n destination vectors from a staged tile whose words start Q words +
// r bits before the destination alignment (Q, r from the source address).
template <int Q>
__device__ __forceinline__ void shifted_copy(uint4* d4, uint32_t buf, int n, int ctid, int nct,
                                             uint32_t r) {
#pragma unroll 2
  for (int k = ctid; k < n; k += nct)
    d4[k] = realign<Q>(lds128(buf + 16u * k), lds128(buf + 16u * k + 16u), r);
}

__global__ void __launch_bounds__(kA2avThreads, BRA_A2AV_MIN_CTAS)
a2av_kernel(const __grid_constant__ A2avArgs a) {
  extern __shared__ __align__(128) uint8_t ring[];   // kStages x kStageStride
  // The P x P counts (row stride P + 1) live in the ring's memory: they are
  // dead before the first chunk is staged.
  int64_t* const s_sc = reinterpret_cast<int64_t*>(ring);
  __shared__ int64_t s_row[kA2avMaxP];   // row i of the counts
  __shared__ int64_t s_sd[kA2avMaxP];    // send displacement of rank i to j
  __shared__ int64_t s_rd[kA2avMaxP];    // receive displacement of i at j
  __shared__ int64_t s_part[2][kA2avThreads];   // column partial sums per row group
  // This CTA's share of rank i's send buffer, cut at destination
  // boundaries: one piece per destination j (possibly empty).
  __shared__ const char* s_src[kA2avMaxP];   // first source byte of the piece
  __shared__ char* s_dst[kA2avMaxP];         // first destination byte
  __shared__ int64_t s_nvec[kA2avMaxP];      // 16-byte destination vectors
  __shared__ int s_head[kA2avMaxP];          // bytes before the first vector
  __shared__ int s_tail[kA2avMaxP];          // bytes after the last vector
  __shared__ int s_list[kA2avMaxP];          // non-empty pieces, in source order
  __shared__ char* s_outp[kA2avMaxP];        // a.out, indexable per lane
  __shared__ int s_nul[kA2avMaxP];           // bit 0: in[r] NULL, bit 1: out[r] NULL
  __shared__ __align__(8) uint64_t s_full[kStages];
  __shared__ __align__(8) uint64_t s_empty[kStages];
  __shared__ int s_npieces;
  __shared__ int s_bad;
  __shared__ int s_abort;

  const int P = a.P;
  const int i = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Loads first: this thread's share of the count matrix (all of it is
  // issued before any is used, so it costs one memory round trip), while
  // thread 0 sets up the barriers.
  int64_t v[kCountIters];
#pragma unroll
  for (int m = 0; m < kCountIters; ++m) {
    const int k = tid + m * kA2avThreads;
    v[m] = k < P * P ? __ldg(a.sc + k) : 0;
  }
  if (tid == 0) {
    s_bad = 0;
    s_abort = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&s_full[s]), 1);
      mbar_init(smem_u32(&s_empty[s]), kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Per-rank pointers into shared memory once: kernel-parameter arrays read
  // with a different index per lane serialise across the warp.
  if (tid < P) {
    char* o = static_cast<char*>(a.out[tid]);
    s_outp[tid] = o;
    s_nul[tid] = (a.in[tid] == nullptr ? 1 : 0) | (o == nullptr ? 2 : 0);
  }
  // Row i straight from global memory: its prefix sums are the send
  // displacements, and its total fixes this CTA's source range, whose start
  // is prefetched into L2 while the rest of the set-up runs.
  if (warp == kRowWarp) {
    const int64_t* row = a.sc + (int64_t)i * P;
    const int64_t r0 = lane < P ? __ldg(row + lane) : 0;
    const int64_t r1 = lane + 32 < P ? __ldg(row + lane + 32) : 0;
    int64_t e0, e1, tot;
    warp_exscan64(r0, r1, lane, e0, e1, tot);
    if (lane < P) {
      s_sd[lane] = e0;
      s_row[lane] = r0;
    }
    if (lane + 32 < P) {
      s_sd[lane + 32] = e1;
      s_row[lane + 32] = r1;
    }
    const bool row_ok = __all_sync(kFull, r0 >= 0 && r1 >= 0);
    if (kPrefetchBytes > 0 && lane == 0 && row_ok && a.in[i] != nullptr) {
      const int64_t lo = split_point(tot, gridDim.x, blockIdx.x);
      int64_t hi = split_point(tot, gridDim.x, blockIdx.x + 1);
      const uintptr_t base = reinterpret_cast<uintptr_t>(a.in[i]);
      const uintptr_t b0 = (base + (uintptr_t)(lo * a.esize) + 15) & ~(uintptr_t)15;
      uintptr_t b1 = (base + (uintptr_t)(hi * a.esize)) & ~(uintptr_t)15;
      if (b1 > b0 + kPrefetchBytes) b1 = b0 + kPrefetchBytes;
      if (b1 > b0) l2_prefetch(reinterpret_cast<const void*>(b0), (uint32_t)(b1 - b0));
    }
  }
  __syncthreads();
  const int ld = P + 1;   // padded row stride: column reads hit distinct banks
  {
    // (src, dst) of entry tid + m * kA2avThreads, stepped without dividing.
    const int step_rows = kA2avThreads / P, step_cols = kA2avThreads - step_rows * P;
    int src = tid / P, dst = tid - (tid / P) * P;
#pragma unroll
    for (int m = 0; m < kCountIters; ++m) {
      const int k = tid + m * kA2avThreads;
      if (m > 0) {
        src += step_rows;
        dst += step_cols;
        if (dst >= P) {
          dst -= P;
          ++src;
        }
      }
      if (k < P * P) {
        s_sc[src * ld + dst] = v[m];
        // A negative count, or a count that would read or write a NULL buffer.
        if (v[m] < 0 || (v[m] > 0 && ((s_nul[src] & 1) | (s_nul[dst] & 2)))) s_bad = 1;
      }
    }
  }
  __syncthreads();

  // Bookkeeping: the sums of column j over source rows k < i (rank i's
  // receive displacement at j) and over all rows (what j receives), as
  // G = blockDim / P groups of threads each summing every G-th row, then
  // one combine per column.
  const int G = blockDim.x / P;   // >= 4 (P <= 64)
  if (tid < G * P) {
    const int j = tid % P, g = tid / P;
    int64_t before = 0, all = 0;
    for (int k = g; k < P; k += G) {
      const int64_t v = s_sc[k * ld + j];
      all += v;
      if (k < i) before += v;
    }
    s_part[0][g * P + j] = before;
    s_part[1][g * P + j] = all;
  }
  __syncthreads();
  if (tid < P) {
    int64_t before = 0, all = 0;
    for (int g = 0; g < G; ++g) {
      before += s_part[0][g * P + tid];
      all += s_part[1][g * P + tid];
    }
    s_rd[tid] = before;
    // Checked variant: a receive total over capacity (every CTA decides alike).
    if (a.check_cap && all > a.cap[tid]) s_bad = 1;
  }
  __syncthreads();
  const bool bad = s_bad != 0;
  if (a.status && blockIdx.x == 0 && i == 0 && tid == 0)
    *a.status = bad ? BRA_ERR_INVALID : BRA_OK;
  if (bad) return;

  if (blockIdx.x == 0) {
    for (int j = tid; j < P; j += blockDim.x) {
      a.sd[(int64_t)i * P + j] = s_sd[j];
      a.rc[(int64_t)j * P + i] = s_row[j];
      a.rd[(int64_t)j * P + i] = s_rd[j];
    }
  }

  // This CTA's contiguous range: equal range blockIdx.x of gridDim.x over
  // rank i's send buffer.
  const int64_t total = s_sd[P - 1] + s_row[P - 1];
  const int64_t lo = split_point(total, gridDim.x, blockIdx.x);
  const int64_t hi = split_point(total, gridDim.x, blockIdx.x + 1);
  const int64_t es = a.esize;

  if (warp == 0) {
    bool has[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = lane + 32 * h;
      has[h] = false;
      if (j < P) {
        const int64_t seg_lo = s_sd[j], seg_hi = seg_lo + s_row[j];
        const int64_t c0 = lo > seg_lo ? lo : seg_lo;
        const int64_t c1 = hi < seg_hi ? hi : seg_hi;
        const int64_t n = c1 > c0 ? (c1 - c0) * es : 0;
        const char* src = static_cast<const char*>(a.in[i]) + (n ? c0 * es : 0);
        char* dst = s_outp[j] + (n ? (s_rd[j] + (c0 - seg_lo)) * es : 0);
        int64_t head = (16 - (int64_t)((uintptr_t)dst & 15)) & 15;
        if (head > n) head = n;
        s_src[j] = src;
        s_dst[j] = dst;
        s_head[j] = (int)head;
        s_nvec[j] = (n - head) >> 4;
        s_tail[j] = (int)((n - head) & 15);
        has[h] = n > 0;
      }
    }
    // Compact list of the non-empty pieces, in source order.
    const unsigned m0 = __ballot_sync(kFull, has[0]);
    const unsigned m1 = __ballot_sync(kFull, has[1]);
    const unsigned below = (1u << lane) - 1u;
    if (has[0]) s_list[__popc(m0 & below)] = lane;
    if (has[1]) s_list[__popc(m0) + __popc(m1 & below)] = lane + 32;
    if (lane == 0) s_npieces = __popc(m0) + __popc(m1);
  }
  __syncthreads();

  // The CTA's source bytes [S, E) are contiguous (the send buffer is ordered
  // by destination).  They stream through the ring as chunks of kChunk bytes
  // from G0 (S rounded down to a granule), each staged with one granule past
  // its end, so a destination vector whose first source byte lies in chunk t
  // (the chunk that writes it) has all 16 of its bytes in that stage.
  const int npieces = s_npieces;
  const uintptr_t S = reinterpret_cast<uintptr_t>(a.in[i]) + (uintptr_t)(lo * es);
  const uintptr_t E = reinterpret_cast<uintptr_t>(a.in[i]) + (uintptr_t)(hi * es);
  const uintptr_t G0 = S & ~(uintptr_t)15, G1 = (E + 15) & ~(uintptr_t)15;
  const int64_t ntiles = hi > lo ? (int64_t)((G1 - G0 + kChunk - 1) / kChunk) : 0;
  volatile int* abort_flag = &s_abort;
  const uint32_t ring_base = smem_u32(ring);
  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      // The ring held the counts: order those generic accesses before the
      // bulk copies overwrite it.
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
#pragma unroll 1
      for (int64_t t = 0; t < ntiles; ++t) {
        if (!mbar_wait(smem_u32(&s_empty[stage]), phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const uintptr_t c0 = G0 + (uintptr_t)t * kChunk;
        const uintptr_t ce = c0 + kChunk + 16 < G1 ? c0 + kChunk + 16 : G1;
        const uint32_t fb = smem_u32(&s_full[stage]);
        mbar_expect_tx(fb, (uint32_t)(ce - c0));
        bulk_load(ring_base + stage * kStageStride, reinterpret_cast<const void*>(c0),
                  (uint32_t)(ce - c0), fb);
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
    int q = 0, stage = 0;   // q: first listed piece not yet finished
    uint32_t phase = 0;
#pragma unroll 1
    for (int64_t t = 0; t < ntiles; ++t) {
      const bool waited = mbar_wait(smem_u32(&s_full[stage]), phase, abort_flag);
      if (!__all_sync(kFull, waited)) break;
      const uintptr_t c0 = G0 + (uintptr_t)t * kChunk;
      const uintptr_t c1 = c0 + kChunk < G1 ? c0 + kChunk : G1;   // bytes this chunk writes
      const uint32_t buf = ring_base + stage * kStageStride;      // holds source byte c0 + o at o
#pragma unroll 1
      for (int qq = q; qq < npieces; ++qq) {
        const int j = s_list[qq];
        const uintptr_t ps = reinterpret_cast<uintptr_t>(s_src[j]);
        if (ps >= c1) break;   // starts in a later chunk
        const int64_t head = s_head[j], nvec = s_nvec[j];
        const int tail = s_tail[j];
        char* const dj = s_dst[j];
        // Vectors v whose first source byte base + 16 v lies in [c0, c1).
        const uintptr_t base = ps + (uintptr_t)head;
        const int64_t vlo = base >= c0 ? 0 : (int64_t)((c0 - base + 15) >> 4);
        int64_t vhi = base >= c1 ? 0 : (int64_t)((c1 - base + 15) >> 4);
        if (vhi > nvec) vhi = nvec;
        if (vhi > vlo) {
          const uint32_t o = (uint32_t)(base + (uintptr_t)(vlo * 16) - c0);
          const uint32_t vbuf = buf + (o & ~15u), delta = o & 15u, r = (delta & 3u) * 8u;
          uint4* d4 = reinterpret_cast<uint4*>(dj + head) + vlo;
          const int n = (int)(vhi - vlo);
          switch (delta >> 2) {
            case 0:
              if (r == 0) {
#pragma unroll 2
                for (int k = ctid; k < n; k += nct) d4[k] = lds128(vbuf + 16u * k);
              } else {
                shifted_copy<0>(d4, vbuf, n, ctid, nct, r);
              }
              break;
            case 1: shifted_copy<1>(d4, vbuf, n, ctid, nct, r); break;
            case 2: shifted_copy<2>(d4, vbuf, n, ctid, nct, r); break;
            default: shifted_copy<3>(d4, vbuf, n, ctid, nct, r); break;
          }
        }
        // Head bytes (lanes 0-15) and tail bytes (lanes 16-31) of the first
        // consumer warp, each written by the chunk holding its source byte.
        if (warp == 1) {
          const int b = lane & 15;
          const int64_t off = lane < 16 ? (b < head ? b : -1)
                                        : (b < tail ? head + nvec * 16 + b : -1);
          if (off >= 0) {
            const uintptr_t sb = ps + (uintptr_t)off;
            if (sb >= c0 && sb < c1) dj[off] = (char)lds8(buf + (uint32_t)(sb - c0));
          }
        }
        if (base + (uintptr_t)(nvec * 16) + (uintptr_t)tail > c1) break;   // continues
        q = qq + 1;
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

int a2av_ctas_per_rank(int P) {
  int resident = 0;
  if (a2av_device_setup(&resident) != cudaSuccess || resident < 1) resident = device_sm_count();
  // One wave over the whole GPU: round down, at least one CTA per rank.
  const int c = resident / P;
  return c < 1 ? 1 : c;
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
