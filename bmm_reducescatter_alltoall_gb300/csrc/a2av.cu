// all_to_all_v among P virtual ranks resident on one GPU, launched on
// exactly the admitted block count.
//
// Semantics ("LowerL2TensorCollectives Pass", 行为 / ABI; addressing as in
// the meta ncclx alltoallv of "vccl alltoallv dev log", 5. ref): rank i sends
// send_counts[i][j] elements to rank j; displacements are exclusive prefix
// sums in element units, over destinations for the sender and over sources
// for the receiver.
//
// Launch width ("LowerL2TensorCollectives Pass", 启动宽度): the call admits
// B = CalAllToAllVBlocks(P, L) blocks, all resident at once.  Here a block is
// one CTA that takes a whole SM (its shared memory leaves room for no second
// CTA), so the exchange occupies exactly min(B, SMs) SMs and leaves the rest
// of the GPU to concurrent work.  The blocks split the whole exchange -- the
// send buffers of ranks 0..P-1 one after another, T elements in all -- into
// equal element ranges: block b copies [b T / nb, (b + 1) T / nb).  A range
// is cut into segments at the source-rank boundaries, and a segment into
// pieces at the destination boundaries (a piece: its 16-byte-aligned
// destination vectors plus head and tail bytes).
//
// Set-up (all warps): the P x P counts go to shared memory; row totals, the
// argument checks (a negative count, a non-zero count that would touch a
// NULL buffer, a receive total over capacity in the checked variant) and
// the segments follow from them.  Every block sees the same matrix, so all
// take the same verdict without a grid sync; a rejected call copies
// nothing.
// Copy: the block's source bytes are cut into chunks of `chunk` bytes
// (16-byte granules; each chunk is staged with one granule more, so every
// destination vector whose first byte lies in a chunk is whole in its
// stage).  Chunk t belongs to warp t mod kWarps, and each warp is its own
// pipeline: lane 0 streams the warp's chunks into the warp's private ring of
// `stages` slots with cp.async.bulk (completion on the slot's mbarrier),
// the warp writes every destination vector of the chunk, shifting the
// staged words into destination alignment (int8 can be off by any byte,
// fp32 by whole words), and lane 0 refills the slot with the warp's chunk
// `stages` later.  One issuing thread per warp: a thread's bulk copies
// complete at about one chunk per load latency, and a warp's own chunk work
// is a chain of dependent steps, so many independent warp pipelines keep an
// SM's loads and stores in flight.  Piece tables are built by all threads,
// kMaxSeg segments at a time.  The head and tail bytes of each piece (before
// its first and after its last 16-byte-aligned destination vector) are
// copied straight from the send buffer, and the bookkeeping (send
// displacements, receive counts, receive displacements) is written, by every
// thread after its warp's first chunk, while the warp's next chunks are in
// flight; the bookkeeping entries are spread over all blocks.
// A granule holding a byte of a buffer never crosses a page the buffer does
// not touch, so granule-wide loads stay in bounds.  Every wait is bounded
// (about 2 s by %globaltimer); a wait that runs out records BRA_ERR_TIMEOUT
// in this file's device word and flags the CTA; every warp then skips its
// remaining chunks (still meeting the CTA barriers) and gives the copies it
// issued time to land before the CTA ends.
#include <cstdint>
#include <mutex>

#include "bra_internal.h"

namespace bra {

__device__ int32_t g_a2av_fault_word = 0;

namespace {

constexpr unsigned kFull = 0xffffffffu;
#ifndef BRA_A2AV_WARPS
#define BRA_A2AV_WARPS 16
#endif
#ifndef BRA_A2AV_MAX_STAGES
#define BRA_A2AV_MAX_STAGES 3
#endif
constexpr int kWarps = BRA_A2AV_WARPS;           // copy warps = pipelines per block
constexpr int kThreads = 32 * kWarps;
constexpr int kRowsPerWarp = (kA2avMaxP + kWarps - 1) / kWarps;   // count rows per warp at set-up
constexpr int kMaxStages = BRA_A2AV_MAX_STAGES;  // ring slots per warp
constexpr int kMaxSeg = 4;                       // segments whose pieces are tabled at once
// Chunk sizes, largest first: the launch takes the first whose ring of at
// least two slots per warp fits beside the P x P counts.  6 KiB chunks in
// two slots ran the bench workload ~5% faster than 4 KiB in three on 64 and
// 128 blocks (fewer chunks, less per-chunk work), and ~7% slower on
// exchanges of a few MB.
constexpr uint32_t kChunks[2] = {6144, 4096};
constexpr uint32_t kSlotPad = 128;               // a chunk is staged with one granule more
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;
static_assert(kThreads >= kMaxSeg * kA2avMaxP, "one thread per tabled piece");
static_assert(kWarps >= kMaxSeg, "one compacting warp per tabled segment");
static_assert(kChunks[0] % 512 == 0 && kChunks[1] % 512 == 0, "chunks: whole 512-byte steps");

// One piece of a segment: its 16-byte-aligned destination vectors, and the
// head and tail bytes before the first and after the last of them.
struct Run {
  uintptr_t vb;      // source address of the first vector's first byte
  char* d;           // destination of the first vector (16-byte aligned)
  int64_t nvec;      // vectors (the piece is listed for the chunk loop when > 0)
  uint8_t delta;     // vb % 16: offset of the staged words from destination alignment
  uint8_t head;      // bytes before the first vector
  uint8_t tail;      // bytes after the last vector
};

__device__ __forceinline__ int64_t warp_sum64(int64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Exclusive scan of 64 values held as (lane, lane + 32) by one warp.
__device__ __forceinline__ void warp_exscan64(int64_t v0, int64_t v1, int lane, int64_t& ex0,
                                              int64_t& ex1, int64_t& total) {
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
// funnel-shifted with word Q + k + 1.
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

// Start of equal range b of nb over n elements (ranges differ by at most one).
__device__ __forceinline__ int64_t split_point(int64_t n, int64_t nb, int64_t b) {
  const int64_t q = n / nb, rem = n - q * nb;
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
// Bounded wait for the phase with the given parity.  False when the CTA was
// flagged by another role or the wait ran out (then this call flags the CTA
// and records BRA_ERR_TIMEOUT in the device word).
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                            volatile int* abort_flag) {
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
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_try(bar, parity) || mbar_wait_slow(bar, parity, abort_flag);
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

#ifndef BRA_A2AV_UNROLL
#define BRA_A2AV_UNROLL 4
#endif
// Copy n destination vectors from a staged tile whose words start Q words +
// r bits before the destination alignment (SHIFT false: the tile is in
// destination alignment), by one warp: lane l takes vectors l, l + 32, ...
// A lane loads its vector's first staged granule and takes the words it
// needs of the next granule from the next lane (lane 31 loads that granule
// itself): one shared-memory granule per vector.  Each lane issues the
// loads of kUnroll vectors before the first store, so their latencies
// overlap.
constexpr int kUnroll = BRA_A2AV_UNROLL;
template <int Q, bool SHIFT>
__device__ __forceinline__ void vec_copy(uint4* d4, uint32_t buf, int n, int lane, uint32_t r) {
  if constexpr (!SHIFT) {
    int k = lane;
#pragma unroll 1
    for (; k + (kUnroll - 1) * 32 < n; k += kUnroll * 32) {
      uint4 a[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) a[u] = lds128(buf + 16u * (uint32_t)(k + u * 32));
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) d4[k + u * 32] = a[u];
    }
#pragma unroll 1
    for (; k < n; k += 32) d4[k] = lds128(buf + 16u * (uint32_t)k);
  } else {
#pragma unroll 1
    for (int base = 0; base < n; base += kUnroll * 32) {
      uint4 a[kUnroll], nx[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int k = base + u * 32 + lane;
        const uint32_t ad = buf + 16u * (uint32_t)k;
        // Granule k: vector k's first, and the second of vector k - 1 (k <= n).
        a[u] = k <= n ? lds128(ad) : make_uint4(0u, 0u, 0u, 0u);
        nx[u] = (lane == 31 && k < n) ? lds128(ad + 16u) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int k = base + u * 32 + lane;
        uint4 b;
        b.x = __shfl_down_sync(kFull, a[u].x, 1);
        b.y = Q >= 1 ? __shfl_down_sync(kFull, a[u].y, 1) : 0u;
        b.z = Q >= 2 ? __shfl_down_sync(kFull, a[u].z, 1) : 0u;
        b.w = Q >= 3 ? __shfl_down_sync(kFull, a[u].w, 1) : 0u;
        if (lane == 31) b = nx[u];
        if (k < n) d4[k] = realign<Q>(a[u], b, r);
      }
    }
  }
}

// Write the vectors of the runs of one staged chunk: vectors whose first
// source byte lies in [c0, c1), held at buf (source byte c0 + o at buf + o,
// plus one granule past c1), by one warp.  q is the warp's first unfinished
// run of the segment; runs are in source order.
__device__ __forceinline__ void copy_runs(const Run* runs, const int* list, int nr, int& q,
                                          uintptr_t c0, uintptr_t c1, uint32_t buf, int lane) {
#pragma unroll 1
  for (int qq = q; qq < nr; ++qq) {
    const Run& rr = runs[list[qq]];
    const uintptr_t vb = rr.vb;
    if (vb >= c1) break;   // starts in a later chunk
    const int64_t nvec = rr.nvec;
    const uintptr_t last = vb + (uintptr_t)((nvec - 1) * 16);   // last vector's first byte
    if (last < c0) {       // ended in a chunk another warp took
      q = qq + 1;
      continue;
    }
    const int64_t vlo = vb >= c0 ? 0 : (int64_t)((c0 - vb + 15) >> 4);
    int64_t vhi = (int64_t)((c1 - vb + 15) >> 4);
    if (vhi > nvec) vhi = nvec;
    const uint32_t o = (uint32_t)(vb + (uintptr_t)(vlo * 16) - c0);
    const uint32_t vbuf = buf + (o & ~15u), delta = rr.delta, r = (delta & 3u) * 8u;
    uint4* d4 = reinterpret_cast<uint4*>(rr.d) + vlo;
    const int n = (int)(vhi - vlo);
    switch (delta >> 2) {
      case 0:
        if (r == 0)
          vec_copy<0, false>(d4, vbuf, n, lane, 0u);
        else
          vec_copy<0, true>(d4, vbuf, n, lane, r);
        break;
      case 1: vec_copy<1, true>(d4, vbuf, n, lane, r); break;
      case 2: vec_copy<2, true>(d4, vbuf, n, lane, r); break;
      default: vec_copy<3, true>(d4, vbuf, n, lane, r); break;
    }
    if (last >= c1) break;   // continues in a later chunk
    q = qq + 1;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
a2av_kernel(const __grid_constant__ A2avArgs a) {
  extern __shared__ __align__(128) uint8_t dyn[];   // ring, then the P x P counts
  __shared__ const char* s_in[kA2avMaxP];
  __shared__ char* s_out[kA2avMaxP];
  __shared__ int64_t s_rowtot[kA2avMaxP];
  // Segments of this block's range, in source order: rank, element range in
  // the rank's send buffer, granule range, and the first chunk of each.
  __shared__ int s_seg_rank[kA2avMaxP];
  __shared__ int64_t s_seg_lo[kA2avMaxP], s_seg_hi[kA2avMaxP];
  __shared__ uintptr_t s_seg_g0[kA2avMaxP], s_seg_g1[kA2avMaxP];
  __shared__ int64_t s_chbase[kA2avMaxP + 1];
  __shared__ Run s_run[kMaxSeg][kA2avMaxP];
  __shared__ int s_list[kMaxSeg][kA2avMaxP];   // runs with vectors, in source order
  __shared__ uint8_t s_has[kMaxSeg][kA2avMaxP];
  __shared__ int s_np[kMaxSeg];
  __shared__ __align__(8) uint64_t s_full[kWarps][kMaxStages];   // each warp's ring slots
  __shared__ int s_nseg;
  __shared__ int s_abort;   // a bounded wait ran out

  const int P = a.P, stages = a.stages;
  const uint32_t chunk = a.chunk, stride = a.chunk + kSlotPad;   // slot bytes
  const int nb = gridDim.x, b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t es = a.esize;
  int64_t* cnt = reinterpret_cast<int64_t*>(dyn + kWarps * stages * stride);
  const uint32_t ring_base = smem_u32(dyn);

  // ---------------- set-up (all warps) ----------------
  if (tid < P) {
    s_in[tid] = static_cast<const char*>(a.in[tid]);
    s_out[tid] = static_cast<char*>(a.out[tid]);
  }
  if (tid == 0) s_abort = 0;
  if (lane < stages) mbar_init(smem_u32(&s_full[warp][lane]), 1);   // the warp's own slots
  __syncwarp();
  if (lane == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  // Rows warp, warp + kWarps, ... of the counts, all loaded before any is
  // used: to shared memory, their totals, and the checks (a negative count,
  // a non-zero count that would touch a NULL buffer; the host marks NULL
  // buffers in two bit masks).
  int bad = 0;
  {
    int64_t v[kRowsPerWarp][2];
#pragma unroll
    for (int m = 0; m < kRowsPerWarp; ++m) {
      const int r = warp + m * kWarps;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = lane + 32 * h;
        v[m][h] = (r < P && j < P) ? __ldg(a.sc + r * P + j) : 0;
      }
    }
#pragma unroll
    for (int m = 0; m < kRowsPerWarp; ++m) {
      const int r = warp + m * kWarps;
      if (r >= P) break;
      const bool in_nul = (a.in_null >> r) & 1u;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = lane + 32 * h;
        if (j < P) {
          const int64_t c = v[m][h];
          cnt[r * P + j] = c;
          bad |= c < 0 || (c > 0 && (in_nul || ((a.out_null >> j) & 1u)));
        }
      }
      const int64_t s = warp_sum64(v[m][0] + v[m][1]);
      if (lane == 0) s_rowtot[r] = s;
    }
  }
  bad = __syncthreads_or(bad);
  // Checked variant: receive totals over capacity (every block decides
  // alike), by warps 2 and 3 while warp 0 lays out the segments.
  int over = 0;
  if (a.check_cap && tid >= 64 && tid < 64 + P) {
    const int j = tid - 64;
    int64_t s = 0;
    for (int k = 0; k < P; ++k) s += cnt[k * P + j];
    over = s > a.cap[j];
  }
  if (warp == 0) {
    // Rank offsets in the concatenated send buffers, this block's range and
    // its segments (compacted, in rank order), and their chunk counts.
    const int64_t v0 = lane < P ? s_rowtot[lane] : 0;
    const int64_t v1 = lane + 32 < P ? s_rowtot[lane + 32] : 0;
    int64_t o0, o1, T;
    warp_exscan64(v0, v1, lane, o0, o1, T);
    const int64_t lo = split_point(T, nb, b), hi = split_point(T, nb, b + 1);
    bool has[2];
    int64_t slo[2], shi[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t off = h ? o1 : o0, tot = h ? v1 : v0;
      has[h] = tot > 0 && off < hi && off + tot > lo;
      slo[h] = lo > off ? lo - off : 0;
      shi[h] = hi - off < tot ? hi - off : tot;
    }
    const unsigned m0 = __ballot_sync(kFull, has[0]);
    const unsigned m1 = __ballot_sync(kFull, has[1]);
    const unsigned below = (1u << lane) - 1u;
    const int nseg = __popc(m0) + __popc(m1);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (!has[h]) continue;
      const int r = lane + 32 * h;
      const int k = h ? __popc(m0) + __popc(m1 & below) : __popc(m0 & below);
      const uintptr_t base = reinterpret_cast<uintptr_t>(s_in[r]);
      s_seg_rank[k] = r;
      s_seg_lo[k] = slo[h];
      s_seg_hi[k] = shi[h];
      s_seg_g0[k] = (base + (uintptr_t)(slo[h] * es)) & ~(uintptr_t)15;
      s_seg_g1[k] = (base + (uintptr_t)(shi[h] * es) + 15) & ~(uintptr_t)15;
    }
    __syncwarp();
    // Chunks per segment and their exclusive prefix (the global chunk index
    // of each segment's first chunk).
    int64_t n0 = 0, n1 = 0;
    if (lane < nseg) n0 = (int64_t)((s_seg_g1[lane] - s_seg_g0[lane] + chunk - 1) / chunk);
    if (lane + 32 < nseg)
      n1 = (int64_t)((s_seg_g1[lane + 32] - s_seg_g0[lane + 32] + chunk - 1) / chunk);
    int64_t e0, e1, nch;
    warp_exscan64(n0, n1, lane, e0, e1, nch);
    if (lane < nseg) s_chbase[lane] = e0;
    if (lane + 32 < nseg) s_chbase[lane + 32] = e1;
    if (lane == 0) {
      s_chbase[nseg] = nch;
      s_nseg = nseg;
    }
  }
  // The last CTA-wide barrier: roles split from here.
  over = __syncthreads_or(over);
  if (a.status && b == 0 && tid == 0) *a.status = (bad || over) ? BRA_ERR_INVALID : BRA_OK;
  if (bad || over) return;   // nothing issued yet: no copy in flight
  volatile int* abort_flag = &s_abort;
  const int nseg = s_nseg;
  const int64_t nch = s_chbase[nseg];

  // ---------------- the warp's pipeline ----------------
  // Lane 0 loads the warp's chunks t = warp, warp + kWarps, ... in order,
  // chunk number i of the warp into slot i % stages; `stages` are loaded
  // up front and each one consumed frees its slot for the next.
  const uint32_t ring = ring_base + (uint32_t)(warp * stages * stride);
  int64_t t_load = warp;
  int sg_load = 0;
  auto load_next = [&](int slot) {
    if (t_load >= nch) return;
    while (s_chbase[sg_load + 1] <= t_load) ++sg_load;
    const uintptr_t c0 = s_seg_g0[sg_load] + (uintptr_t)(t_load - s_chbase[sg_load]) * chunk;
    const uintptr_t G1 = s_seg_g1[sg_load];
    const uintptr_t ce = c0 + chunk + 16 < G1 ? c0 + chunk + 16 : G1;
    const uint32_t fb = smem_u32(&s_full[warp][slot]);
    mbar_expect_tx(fb, (uint32_t)(ce - c0));
    bulk_load(ring + slot * stride, reinterpret_cast<const void*>(c0), (uint32_t)(ce - c0),
              fb);
    t_load += kWarps;
  };
  if (lane == 0)
    for (int k = 0; k < stages; ++k) load_next(k);

  // Bookkeeping, entries (i, j) dealt round-robin over the blocks, then over
  // each block's threads; every thread does its share after its warp's first
  // chunk (below), while the warp's next chunks are in flight.
  auto bookkeeping = [&]() {
    const int64_t PP = (int64_t)P * P;
#pragma unroll 1
    for (int64_t e = b + (int64_t)nb * tid; e < PP; e += (int64_t)nb * kThreads) {
      const int i = (int)(e / P), j = (int)(e % P);
      int64_t sd = 0, rd = 0;
      for (int k = 0; k < j; ++k) sd += cnt[i * P + k];
      for (int k = 0; k < i; ++k) rd += cnt[k * P + j];
      a.sd[(int64_t)i * P + j] = sd;
      a.rc[(int64_t)j * P + i] = cnt[i * P + j];
      a.rd[(int64_t)j * P + i] = rd;
    }
  };
  bool book_done = false;

  bool live = true;
  int slot = 0;
  uint32_t ph = 0;
  int64_t t = warp;   // the warp's next chunk to write
  int sg = 0, q = 0;  // its segment and first unfinished run there
#pragma unroll 1
  for (int b0 = 0; b0 < nseg; b0 += kMaxSeg) {
    const int nbatch = nseg - b0 < kMaxSeg ? nseg - b0 : kMaxSeg;
    if (b0 > 0) __syncthreads();   // every warp is done with the previous tables
    // Piece (s, j) of segment b0 + s by thread s * 64 + j.
    if (tid < nbatch * kA2avMaxP) {
      const int s = tid / kA2avMaxP, j = tid % kA2avMaxP;
      Run& rr = s_run[s][j];
      rr.nvec = 0;
      rr.head = 0;
      rr.tail = 0;
      if (j < P) {
        const int sgi = b0 + s, i = s_seg_rank[sgi];
        int64_t sd = 0, rd = 0;
#pragma unroll 8
        for (int k = 0; k < j; ++k) sd += cnt[i * P + k];
#pragma unroll 8
        for (int k = 0; k < i; ++k) rd += cnt[k * P + j];
        const int64_t c = cnt[i * P + j], lo = s_seg_lo[sgi], hi = s_seg_hi[sgi];
        const int64_t c0 = lo > sd ? lo : sd;
        const int64_t c1 = hi < sd + c ? hi : sd + c;
        const int64_t n = c1 > c0 ? (c1 - c0) * es : 0;
        if (n > 0) {
          const char* src = s_in[i] + c0 * es;
          char* dst = s_out[j] + (rd + (c0 - sd)) * es;
          int64_t head = (16 - (int64_t)((uintptr_t)dst & 15)) & 15;
          if (head > n) head = n;
          rr.vb = reinterpret_cast<uintptr_t>(src) + (uintptr_t)head;
          rr.d = dst + head;
          rr.nvec = (n - head) >> 4;
          rr.delta = (uint8_t)(rr.vb & 15u);
          rr.head = (uint8_t)head;
          rr.tail = (uint8_t)((n - head) & 15);
        }
      }
      s_has[s][j] = rr.nvec > 0 ? 1 : 0;
    }
    __syncthreads();
    // Compact list of each segment's pieces with vectors (warp s).
    if (warp < nbatch) {
      const int s = warp;
      const bool h0 = lane < P && s_has[s][lane];
      const bool h1 = lane + 32 < P && s_has[s][lane + 32];
      const unsigned m0 = __ballot_sync(kFull, h0);
      const unsigned m1 = __ballot_sync(kFull, h1);
      const unsigned below = (1u << lane) - 1u;
      if (h0) s_list[s][__popc(m0 & below)] = lane;
      if (h1) s_list[s][__popc(m0) + __popc(m1 & below)] = lane + 32;
      if (lane == 0) s_np[s] = __popc(m0) + __popc(m1);
    }
    __syncthreads();
    // Head and tail bytes of the batch's pieces, straight from the send
    // buffer: byte slot x = (piece, b) with b < 15 the head's byte b and
    // 16 <= b < 31 the tail's byte b - 16, dealt over every thread, four
    // loads in flight per thread.  Each warp does its share after writing
    // its first chunk of the batch, while its next chunks are in flight.
    auto head_tail = [&]() {
      const int nslot = nbatch * kA2avMaxP * 32;
#pragma unroll 1
      for (int x0 = 0; x0 < nslot; x0 += 4 * kThreads) {
        char v[4];
        char* dst[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int x = x0 + u * kThreads + tid;
          dst[u] = nullptr;
          v[u] = 0;
          if (x < nslot) {
            const Run& rr = s_run[(x >> 5) / kA2avMaxP][(x >> 5) % kA2avMaxP];
            const int bb = x & 31;
            const bool in_head = bb < rr.head;
            const bool in_tail = bb >= 16 && bb - 16 < rr.tail;
            if (in_head || in_tail) {
              const int64_t o = in_head ? (int64_t)bb - rr.head : rr.nvec * 16 + (bb - 16);
              v[u] = __ldg(reinterpret_cast<const char*>(rr.vb) + o);
              dst[u] = rr.d + o;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (dst[u]) *dst[u] = v[u];
      }
    };
    bool ht_done = false;

    // The warp's chunks of this batch.
    const int64_t te = s_chbase[b0 + nbatch];
#pragma unroll 1
    for (; t < te && live; t += kWarps) {
      while (s_chbase[sg + 1] <= t) {
        ++sg;
        q = 0;
      }
      const bool waited = mbar_wait(smem_u32(&s_full[warp][slot]), ph, abort_flag);
      live = __all_sync(kFull, waited);
      if (!live) break;
      const uintptr_t c0 = s_seg_g0[sg] + (uintptr_t)(t - s_chbase[sg]) * chunk;
      const uintptr_t G1 = s_seg_g1[sg];
      const uintptr_t c1 = c0 + chunk < G1 ? c0 + chunk : G1;   // bytes this chunk writes
      const int s = sg - b0;
      copy_runs(s_run[s], s_list[s], s_np[s], q, c0, c1, ring + slot * stride, lane);
      __syncwarp();
      if (lane == 0) load_next(slot);   // the warp's chunk `stages` later
      if (++slot == stages) {
        slot = 0;
        ph ^= 1u;
      }
      if (!ht_done) {
        head_tail();
        ht_done = true;
        if (!book_done) {
          bookkeeping();
          book_done = true;
        }
      }
    }
    if (live && !ht_done) head_tail();   // the warp had no chunk in this batch
  }
  if (live && !book_done) bookkeeping();
  if (!live) {   // a wait ran out: give copies already issued time to land
    if (lane == 0) {
      const unsigned long long t0 = global_ns();
      while (global_ns() - t0 < 2000000ull) {
      }
    }
    return;
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
    const bool done = mbar_wait(smem_u32(&bar), 0, &abort_flag);
    *status = done ? BRA_OK : BRA_ERR_TIMEOUT;
  }
}

// Per device: SM count, and the shared memory a block may take.
struct A2avDeviceInfo {
  bool ready = false;
  int sms = 0;
  int dyn_max = 0;   // dynamic shared memory per block (opt-in maximum less the static part)
};

cudaError_t a2av_device_info(A2avDeviceInfo* out) {
  static std::mutex mu;
  static A2avDeviceInfo info[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  A2avDeviceInfo& di = info[dev & 63];
  if (!di.ready) {
    int sms = 0, optin = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
        cudaSuccess)
      return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, a2av_kernel)) != cudaSuccess) return e;
    di.dyn_max = optin - (int)fa.sharedSizeBytes;
    if ((e = cudaFuncSetAttribute(a2av_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  di.dyn_max)) != cudaSuccess)
      return e;
    di.sms = sms > 0 ? sms : 1;
    di.ready = true;
  }
  *out = di;
  return cudaSuccess;
}

// Chunk size and ring slots per warp for P ranks: the largest chunk of
// kChunks with at least two slots per warp beside the P x P counts, and as
// many slots as fit, at most kMaxStages.  Slots 0 means none fits.
void ring_for(const A2avDeviceInfo& di, int P, uint32_t* chunk, int* slots) {
  const int cnt_bytes = (P * P * 8 + 127) / 128 * 128;
  for (uint32_t c : kChunks) {
    const int s = (di.dyn_max - cnt_bytes) / (kWarps * (int)(c + kSlotPad));
    if (s >= 2) {
      *chunk = c;
      *slots = s > kMaxStages ? kMaxStages : s;
      return;
    }
  }
  *chunk = kChunks[1];
  *slots = 0;
}

}  // namespace

int a2av_launch_blocks(int64_t B) {
  A2avDeviceInfo di;
  if (a2av_device_info(&di) != cudaSuccess) return -1;
  return B < di.sms ? (int)B : di.sms;
}

cudaError_t launch_a2av(const A2avArgs& args, int blocks, cudaStream_t st) {
  A2avDeviceInfo di;
  cudaError_t e = a2av_device_info(&di);
  if (e != cudaSuccess) return e;
  A2avArgs a = args;
  ring_for(di, a.P, &a.chunk, &a.stages);
  if (a.stages < 2 || blocks < 1) return cudaErrorInvalidConfiguration;
  // The whole shared memory a block may take, whatever the ring uses: two
  // blocks never share an SM, and the exchange occupies `blocks` SMs.
  const size_t dyn = (size_t)di.dyn_max;
  a2av_kernel<<<blocks, kThreads, dyn, st>>>(a);
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
