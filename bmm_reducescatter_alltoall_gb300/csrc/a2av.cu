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
//
// A CTA of source rank i takes an equal element range [lo, hi) of rank i's
// send buffer.  That range is contiguous in the source (the buffer is
// ordered by destination) and cut at the destination boundaries into at
// most P pieces; a piece is its 16-byte-aligned destination vectors plus
// head and tail bytes before the first / after the last vector.  Roles:
//   warp 0   reads row i of the counts from global memory, scans it (the
//            send displacements), fixes [lo, hi) and publishes them; lane 0
//            then streams the range through a kStages-deep shared-memory
//            ring in chunks of kChunk bytes (16-byte granules, each chunk
//            staged with one granule of overlap) with cp.async.bulk (TMA
//            bulk copies, completion on an mbarrier), starting before the
//            rest of the set-up is done;
//   warps 1-7 (consumers) read the whole P x P count matrix (P <= 64),
//            each thread a slice of one column, reject the call if any count
//            is negative, a non-zero count would touch a NULL buffer or
//            (checked variant) a receive total is over capacity (every CTA
//            sees the same matrix, so all take the same decision without a
//            grid sync), sum every column below row i (the receive
//            displacements) and over all rows, write the bookkeeping (CTA 0
//            of each rank), build the pieces, tell the producer the verdict,
//            and then, for each chunk, write every vector of every
//            piece whose first source byte lies in the chunk, shifting the
//            words into destination alignment (int8 can be off by any byte,
//            fp32 by whole words), while 32 lanes write the head and tail
//            bytes that lie in it.
// A granule holding a byte of a buffer never crosses a page the buffer does
// not touch, so the granule-wide loads stay in bounds.  If the call is
// rejected the producer waits for the copies it issued before the CTA ends.
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
#define BRA_A2AV_MIN_CTAS 3
#endif
constexpr int kStages = BRA_A2AV_STAGES;
constexpr int kTileVecs = BRA_A2AV_TILE_VECS;            // 16-byte destination vectors
// Source bytes a chunk writes out; it is staged with one granule more.
constexpr uint32_t kChunk = kTileVecs * 16;
constexpr int kStageBytes = kChunk + 16;
constexpr int kStageStride = (kStageBytes + 127) / 128 * 128;
constexpr int kRingBytes = kStages * kStageStride;
#ifndef BRA_A2AV_THREADS
#define BRA_A2AV_THREADS 256
#endif
constexpr int kA2avThreads = BRA_A2AV_THREADS;   // one producer warp + consumer warps
constexpr int kConsumerWarps = kA2avThreads / 32 - 1;
constexpr int kConsumers = kConsumerWarps * 32;
// Count rows per consumer thread: rows g, g + G, ... of one column, with
// G = kConsumers / P >= kConsumers / kA2avMaxP row groups.
constexpr int kColIters = (kA2avMaxP + kConsumers / kA2avMaxP - 1) / (kConsumers / kA2avMaxP);
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
// Bounded wait that does not leave early when another role gave up: used
// where the CTA must still observe the phase (copies in flight, set-up
// hand-offs).  Running out records BRA_ERR_TIMEOUT like mbar_wait.
__device__ __noinline__ bool mbar_wait_plain(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int k = 0; k < 64; ++k)
      if (mbar_try(bar, parity)) return true;
    if (global_ns() - t0 > kWaitTimeoutNs) {
      *abort_flag = 1;
      atomicExch(&g_a2av_fault_word, (int32_t)BRA_ERR_TIMEOUT);
      return false;
    }
  }
}
// Barrier among the consumer warps only (named barrier 1).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
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
  __shared__ int64_t s_row[kA2avMaxP];   // row i of the counts
  __shared__ int64_t s_sd[kA2avMaxP];    // send displacement of rank i to j
  __shared__ int64_t s_rd[kA2avMaxP];    // receive displacement of i at j
  __shared__ int64_t s_part[2][kConsumers];   // column partial sums per row group
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
  __shared__ __align__(8) uint64_t s_row_ready;    // warp 0 has published row i
  __shared__ __align__(8) uint64_t s_setup_done;   // the consumers' verdict (accept / reject)
  __shared__ int64_t s_lo, s_hi;
  __shared__ int s_npieces;
  __shared__ int s_bad;
  __shared__ int s_reject;   // the consumers rejected the call
  __shared__ int s_abort;    // a bounded wait ran out

  const int P = a.P;
  const int i = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ctid = tid - 32;   // consumer thread index (warps 1..7)
  // Consumer thread (j, g) = (ctid % P, ctid / P), ctid < G * P, owns
  // column j of the counts on the rows k = g, g + G, ... (a warp reads whole
  // rows, so the loads coalesce).
  const int G = kConsumers / P;   // >= 3 (P <= 64)
  const int cj = ctid % P, cg = ctid / P;
  const bool col_owner = warp > 0 && ctid < G * P;

  // Loads first, so they overlap the barrier set-up: row i (warp 0) and
  // each consumer thread's share of the count matrix, all issued before any
  // is used.
  int64_t r0 = 0, r1 = 0;
  int64_t v[kColIters];
  if (warp == 0) {
    const int64_t* row = a.sc + (int64_t)i * P;
    r0 = lane < P ? __ldg(row + lane) : 0;
    r1 = lane + 32 < P ? __ldg(row + lane + 32) : 0;
  } else {
#pragma unroll
    for (int m = 0; m < kColIters; ++m) {
      const int k = cg + m * G;
      v[m] = (col_owner && k < P) ? __ldg(a.sc + (int64_t)k * P + cj) : 0;
    }
    // Per-rank pointers into shared memory once: kernel-parameter arrays
    // read with a different index per lane serialise across the warp.
    if (ctid < P) {
      char* o = static_cast<char*>(a.out[ctid]);
      s_outp[ctid] = o;
      s_nul[ctid] = (a.in[ctid] == nullptr ? 1 : 0) | (o == nullptr ? 2 : 0);
    }
  }
  if (tid == 0) {
    s_bad = 0;
    s_reject = 0;
    s_abort = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&s_full[s]), 1);
      mbar_init(smem_u32(&s_empty[s]), kConsumerWarps);
    }
    mbar_init(smem_u32(&s_row_ready), 1);
    mbar_init(smem_u32(&s_setup_done), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();   // the only CTA-wide barrier: roles split from here
  volatile int* abort_flag = &s_abort;
  const uint32_t ring_base = smem_u32(ring);
  const int64_t es = a.esize;

  if (warp == 0) {
    // Row i: its prefix sums are the send displacements, and its total fixes
    // this CTA's source range, which lane 0 starts streaming at once.
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
    const int64_t lo = row_ok ? split_point(tot, gridDim.x, blockIdx.x) : 0;
    const int64_t hi = row_ok ? split_point(tot, gridDim.x, blockIdx.x + 1) : 0;
    __syncwarp();
    if (lane != 0) return;
    s_lo = lo;
    s_hi = hi;
    mbar_arrive(smem_u32(&s_row_ready));

    // Producer.  Nothing is streamed for a row with a negative count or a
    // NULL buffer; the consumers reject such calls.
    const bool go = row_ok && hi > lo && a.in[i] != nullptr;
    const uintptr_t S = go ? reinterpret_cast<uintptr_t>(a.in[i]) + (uintptr_t)(lo * es) : 0;
    const uintptr_t E = go ? reinterpret_cast<uintptr_t>(a.in[i]) + (uintptr_t)(hi * es) : 0;
    const uintptr_t G0 = S & ~(uintptr_t)15, G1 = (E + 15) & ~(uintptr_t)15;
    const int64_t ntiles = go ? (int64_t)((G1 - G0 + kChunk - 1) / kChunk) : 0;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int64_t issued = 0;
#pragma unroll 1
    for (int64_t t = 0; t < ntiles; ++t) {
      // Also leaves when the consumers reject the call (they raise the flag).
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
      ++issued;
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // The CTA may not finish while copies it issued are in flight, so learn
    // the consumers' verdict.  A rejected call consumes nothing (and so no
    // stage was reused): wait for each issued copy to land.
    const bool told = mbar_wait_plain(smem_u32(&s_setup_done), 0, abort_flag);
    if (told && s_reject) {
      for (int s = 0; s < kStages && s < issued; ++s)
        if (!mbar_wait_plain(smem_u32(&s_full[s]), 0, abort_flag)) break;
    } else if (!ok || !told) {   // a wait ran out: give copies already issued time to land
      const unsigned long long t0 = global_ns();
      while (global_ns() - t0 < 2000000ull) {
      }
    }
    return;
  }

  // Consumers (warps 1..7): the checks, the column sums and the pieces,
  // synchronised among themselves by named barrier 1.  Thread (j, g) checks
  // its counts (negative, or non-zero with a NULL buffer at either end) and
  // sums column j over its rows below i (rank i's receive displacement at
  // j) and over all its rows (what j receives); one combine per column.
  if (col_owner) {
    int64_t before = 0, all = 0;
    bool bad_here = false;
    const bool out_nul = (s_nul[cj] & 2) != 0;
#pragma unroll
    for (int m = 0; m < kColIters; ++m) {
      const int k = cg + m * G;
      if (k < P) {
        const int64_t c = v[m];
        all += c;
        if (k < i) before += c;
        bad_here |= c < 0 || (c > 0 && ((s_nul[k] & 1) || out_nul));
      }
    }
    if (bad_here) s_bad = 1;
    s_part[0][cg * P + cj] = before;
    s_part[1][cg * P + cj] = all;
  }
  consumer_sync();
  if (ctid < P) {
    int64_t before = 0, all = 0;
    for (int g = 0; g < G; ++g) {
      before += s_part[0][g * P + ctid];
      all += s_part[1][g * P + ctid];
    }
    s_rd[ctid] = before;
    // Checked variant: a receive total over capacity (every CTA decides alike).
    if (a.check_cap && all > a.cap[ctid]) s_bad = 1;
  }
  // Row i as warp 0 published it (it does so without waiting on anything;
  // one thread observes the hand-off and the barrier spreads it, so a
  // timeout here would send every consumer the same way).
  if (ctid == 0 && !mbar_wait_plain(smem_u32(&s_row_ready), 0, abort_flag)) s_bad = 1;
  consumer_sync();
  const bool bad = s_bad != 0;
  if (a.status && blockIdx.x == 0 && i == 0 && ctid == 0)
    *a.status = bad ? BRA_ERR_INVALID : BRA_OK;
  if (bad) {
    if (ctid == 0) {
      s_reject = 1;
      *abort_flag = 1;   // a producer waiting for a free stage leaves its loop
      mbar_arrive(smem_u32(&s_setup_done));
    }
    return;
  }
  const int64_t lo = s_lo, hi = s_hi;

  if (blockIdx.x == 0) {
    for (int j = ctid; j < P; j += kConsumers) {
      a.sd[(int64_t)i * P + j] = s_sd[j];
      a.rc[(int64_t)j * P + i] = s_row[j];
      a.rd[(int64_t)j * P + i] = s_rd[j];
    }
  }

  if (warp == 1) {
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
  consumer_sync();
  if (ctid == 0) mbar_arrive(smem_u32(&s_setup_done));   // accepted

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
  const int nct = kConsumers;
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

// Diagnostic: one bounded wait (the same helper the exchange uses) on a
// barrier nothing arrives at.  It runs out after kWaitTimeoutNs, records
// BRA_ERR_TIMEOUT in this file's fault word and returns; *status gets the
// outcome.
__global__ void a2av_wait_probe_kernel(int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool done = mbar_wait_plain(smem_u32(&bar), 0, &abort_flag);
    *status = done ? BRA_OK : BRA_ERR_TIMEOUT;
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

cudaError_t launch_a2av_wait_probe(int32_t* status, cudaStream_t st) {
  a2av_wait_probe_kernel<<<1, 32, 0, st>>>(status);
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
