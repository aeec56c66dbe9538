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
// Roles after set-up:
//   warp 0, lane 0   producer: streams the segments' source bytes through a
//                    ring of `stages` chunks of kChunk bytes (16-byte
//                    granules, each chunk staged with one granule more) with
//                    cp.async.bulk (completion on an mbarrier);
//   warps 1..        kGroups consumer groups of kGroupWarps warps; group g
//                    takes chunks g, g + kGroups, ... and writes every vector
//                    whose first source byte lies in the chunk, shifting the
//                    words into destination alignment (int8 can be off by any
//                    byte, fp32 by whole words), while the group's first warp
//                    writes the head and tail bytes that lie in it.  Piece
//                    tables are built kMaxSeg segments at a time.
//   Afterwards the consumers write the bookkeeping (send displacements,
//   receive counts, receive displacements), entries spread over all blocks.
// A granule holding a byte of a buffer never crosses a page the buffer does
// not touch, so granule-wide loads stay in bounds.  Every wait is bounded
// (about 2 s by %globaltimer); a wait that runs out records BRA_ERR_TIMEOUT
// in this file's device word, flags the CTA, and all roles leave their
// loops (the consumers still meet their named barriers).
#include <cstdint>
#include <mutex>

#include "bra_internal.h"

namespace bra {

__device__ int32_t g_a2av_fault_word = 0;

namespace {

constexpr unsigned kFull = 0xffffffffu;
#ifndef BRA_A2AV_GROUPS
#define BRA_A2AV_GROUPS 4
#endif
#ifndef BRA_A2AV_GROUP_WARPS
#define BRA_A2AV_GROUP_WARPS 4
#endif
#ifndef BRA_A2AV_MAX_STAGES
#define BRA_A2AV_MAX_STAGES 12
#endif
constexpr int kGroups = BRA_A2AV_GROUPS;
constexpr int kGroupWarps = BRA_A2AV_GROUP_WARPS;
constexpr int kGroupThreads = 32 * kGroupWarps;
constexpr int kConsumers = kGroups * kGroupThreads;
constexpr int kThreads = 32 + kConsumers;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxStages = BRA_A2AV_MAX_STAGES;
constexpr int kMaxSeg = 4;                       // segments whose pieces are tabled at once
constexpr uint32_t kChunk = 16384;               // source bytes a chunk writes out
constexpr int kStageStride = kChunk + 128;       // staged with one granule more
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;
static_assert(kConsumers >= kMaxSeg * kA2avMaxP, "one consumer thread per tabled piece");
static_assert(kGroups * kGroupWarps >= kMaxSeg, "one compacting warp per tabled segment");
// Chunk t goes to ring stage t % stages and to group t % kGroups.  With the
// stage count a multiple of kGroups every stage belongs to one group, whose
// uses of it are its own consecutive chunks; otherwise a group could wait on
// a stage's full barrier two uses ahead of the load in flight, and the
// parity wait would pass on the older phase.
static_assert(kMaxStages % kGroups == 0, "stages come in whole multiples of the groups");

struct Piece {
  const char* src;   // first source byte
  char* dst;         // first destination byte
  int64_t nvec;      // 16-byte destination vectors
  int head;          // bytes before the first vector
  int tail;          // bytes after the last vector
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
// Bounded wait for the phase with the given parity.  False when the CTA was
// flagged by another role or the wait ran out (then this call flags the CTA
// and records BRA_ERR_TIMEOUT in the device word).
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

#ifndef BRA_A2AV_UNROLL
#define BRA_A2AV_UNROLL 4
#endif
// Copy n destination vectors from a staged tile whose words start Q words +
// r bits before the destination alignment (SHIFT false: the tile is in
// destination alignment).  Each thread issues the shared-memory loads of
// kUnroll vectors before the first store, so their latencies overlap.
constexpr int kUnroll = BRA_A2AV_UNROLL;
template <int Q, bool SHIFT>
__device__ __forceinline__ void vec_copy(uint4* d4, uint32_t buf, int n, int t, uint32_t r) {
  int k = t;
#pragma unroll 1
  for (; k + (kUnroll - 1) * kGroupThreads < n; k += kUnroll * kGroupThreads) {
    uint4 a[kUnroll], b[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t ad = buf + 16u * (uint32_t)(k + u * kGroupThreads);
      a[u] = lds128(ad);
      if (SHIFT) b[u] = lds128(ad + 16u);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      d4[k + u * kGroupThreads] = SHIFT ? realign<Q>(a[u], b[u], r) : a[u];
  }
#pragma unroll 1
  for (; k < n; k += kGroupThreads) {
    const uint32_t ad = buf + 16u * (uint32_t)k;
    d4[k] = SHIFT ? realign<Q>(lds128(ad), lds128(ad + 16u), r) : lds128(ad);
  }
}

// Write the vectors and the head / tail bytes of the pieces of one staged
// chunk: source bytes [c0, c1) held at buf (source byte c0 + o at buf + o,
// plus one granule past c1).  q is the group's first unfinished piece of the
// segment; pieces are in source order.
__device__ __forceinline__ void copy_chunk(const Piece* pc, const int* list, int np, int& q,
                                           uintptr_t c0, uintptr_t c1, uint32_t buf, int gt,
                                           bool head_warp, int lane) {
#pragma unroll 1
  for (int qq = q; qq < np; ++qq) {
    const Piece& p = pc[list[qq]];
    const uintptr_t ps = reinterpret_cast<uintptr_t>(p.src);
    if (ps >= c1) break;   // starts in a later chunk
    const int64_t head = p.head, nvec = p.nvec;
    const int tail = p.tail;
    const uintptr_t base = ps + (uintptr_t)head;
    const uintptr_t pe = base + (uintptr_t)(nvec * 16) + (uintptr_t)tail;
    if (pe <= c0) {        // ended in a chunk another group took
      q = qq + 1;
      continue;
    }
    char* const dj = p.dst;
    // Vectors v whose first source byte base + 16 v lies in [c0, c1).
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
          if (r == 0)
            vec_copy<0, false>(d4, vbuf, n, gt, 0u);
          else
            vec_copy<0, true>(d4, vbuf, n, gt, r);
          break;
        case 1: vec_copy<1, true>(d4, vbuf, n, gt, r); break;
        case 2: vec_copy<2, true>(d4, vbuf, n, gt, r); break;
        default: vec_copy<3, true>(d4, vbuf, n, gt, r); break;
      }
    }
    // Head bytes (lanes 0-15) and tail bytes (lanes 16-31) of the group's
    // first warp, each written by the chunk holding its source byte.
    if (head_warp) {
      const int bb = lane & 15;
      const int64_t off = lane < 16 ? (bb < head ? bb : -1)
                                    : (bb < tail ? head + nvec * 16 + bb : -1);
      if (off >= 0) {
        const uintptr_t sb = ps + (uintptr_t)off;
        if (sb >= c0 && sb < c1) dj[off] = (char)lds8(buf + (uint32_t)(sb - c0));
      }
    }
    if (pe > c1) break;   // continues in a later chunk
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
  __shared__ Piece s_piece[kMaxSeg][kA2avMaxP];
  __shared__ int s_list[kMaxSeg][kA2avMaxP];   // non-empty pieces, in source order
  __shared__ uint8_t s_has[kMaxSeg][kA2avMaxP];
  __shared__ int s_np[kMaxSeg];
  __shared__ __align__(8) uint64_t s_full[kMaxStages];
  __shared__ __align__(8) uint64_t s_empty[kMaxStages];
  __shared__ int s_nseg;
  __shared__ int s_bad;
  __shared__ int s_abort;   // a bounded wait ran out

  const int P = a.P, stages = a.stages;
  const int nb = gridDim.x, b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t es = a.esize;
  int64_t* cnt = reinterpret_cast<int64_t*>(dyn + stages * kStageStride);
  const uint32_t ring_base = smem_u32(dyn);

  // ---------------- set-up (all warps) ----------------
#pragma unroll 4
  for (int k = tid; k < P * P; k += kThreads) cnt[k] = __ldg(a.sc + k);
  if (tid < P) {
    s_in[tid] = static_cast<const char*>(a.in[tid]);
    s_out[tid] = static_cast<char*>(a.out[tid]);
  }
  if (tid == 0) {
    s_bad = 0;
    s_abort = 0;
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&s_full[s]), 1);
      mbar_init(smem_u32(&s_empty[s]), kGroupWarps);   // the warps of the consuming group
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // Row totals and the checks, a warp per row.
  for (int r = warp; r < P; r += kWarps) {
    const bool in_nul = s_in[r] == nullptr;
    int64_t s = 0;
    bool bad = false;
    for (int j = lane; j < P; j += 32) {
      const int64_t c = cnt[r * P + j];
      s += c;
      bad |= c < 0 || (c > 0 && (in_nul || s_out[j] == nullptr));
    }
    s = warp_sum64(s);
    if (__any_sync(kFull, bad) && lane == 0) s_bad = 1;
    if (lane == 0) s_rowtot[r] = s;
  }
  // Checked variant: a receive total over capacity (every block decides alike).
  if (a.check_cap && tid < P) {
    int64_t s = 0;
    for (int k = 0; k < P; ++k) s += cnt[k * P + tid];
    if (s > a.cap[tid]) s_bad = 1;
  }
  __syncthreads();
  const bool bad = s_bad != 0;
  if (a.status && b == 0 && tid == 0) *a.status = bad ? BRA_ERR_INVALID : BRA_OK;
  if (bad) return;   // nothing issued yet: no copy in flight

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
    if (lane < nseg) n0 = (int64_t)((s_seg_g1[lane] - s_seg_g0[lane] + kChunk - 1) / kChunk);
    if (lane + 32 < nseg)
      n1 = (int64_t)((s_seg_g1[lane + 32] - s_seg_g0[lane + 32] + kChunk - 1) / kChunk);
    int64_t e0, e1, nch;
    warp_exscan64(n0, n1, lane, e0, e1, nch);
    if (lane < nseg) s_chbase[lane] = e0;
    if (lane + 32 < nseg) s_chbase[lane + 32] = e1;
    if (lane == 0) {
      s_chbase[nseg] = nch;
      s_nseg = nseg;
    }
  }
  __syncthreads();   // the last CTA-wide barrier: roles split from here
  volatile int* abort_flag = &s_abort;
  const int nseg = s_nseg;

  if (warp == 0) {
    if (lane != 0) return;
    // ---------------- producer ----------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
#pragma unroll 1
    for (int sg = 0; sg < nseg && ok; ++sg) {
      const uintptr_t G0 = s_seg_g0[sg], G1 = s_seg_g1[sg];
#pragma unroll 1
      for (uintptr_t c0 = G0; c0 < G1; c0 += kChunk) {
        if (!mbar_wait(smem_u32(&s_empty[stage]), phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const uintptr_t ce = c0 + kChunk + 16 < G1 ? c0 + kChunk + 16 : G1;
        const uint32_t fb = smem_u32(&s_full[stage]);
        mbar_expect_tx(fb, (uint32_t)(ce - c0));
        bulk_load(ring_base + stage * kStageStride, reinterpret_cast<const void*>(c0),
                  (uint32_t)(ce - c0), fb);
        if (++stage == stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) {   // a wait ran out: give copies already issued time to land
      const unsigned long long t0 = global_ns();
      while (global_ns() - t0 < 2000000ull) {
      }
    }
    return;
  }

  // ---------------- consumers (warps 1..) ----------------
  const int ct = tid - 32;                       // consumer thread
  const int g = ct / kGroupThreads;              // group
  const int gt = ct - g * kGroupThreads;         // thread within the group
  const bool head_warp = gt < 32;
  bool live = true;
#pragma unroll 1
  for (int b0 = 0; b0 < nseg; b0 += kMaxSeg) {
    const int nbatch = nseg - b0 < kMaxSeg ? nseg - b0 : kMaxSeg;
    if (b0 > 0) consumer_sync();   // every group is done with the previous tables
    // Piece (s, j) of segment b0 + s by consumer thread s * 64 + j.
    if (ct < nbatch * kA2avMaxP) {
      const int s = ct / kA2avMaxP, j = ct % kA2avMaxP;
      bool has = false;
      if (j < P) {
        const int sg = b0 + s, i = s_seg_rank[sg];
        int64_t sd = 0, rd = 0;
#pragma unroll 8
        for (int k = 0; k < j; ++k) sd += cnt[i * P + k];
#pragma unroll 8
        for (int k = 0; k < i; ++k) rd += cnt[k * P + j];
        const int64_t c = cnt[i * P + j], lo = s_seg_lo[sg], hi = s_seg_hi[sg];
        const int64_t c0 = lo > sd ? lo : sd;
        const int64_t c1 = hi < sd + c ? hi : sd + c;
        const int64_t n = c1 > c0 ? (c1 - c0) * es : 0;
        Piece& p = s_piece[s][j];
        p.src = s_in[i] + (n ? c0 * es : 0);
        char* dst = s_out[j] + (n ? (rd + (c0 - sd)) * es : 0);
        int64_t head = (16 - (int64_t)((uintptr_t)dst & 15)) & 15;
        if (head > n) head = n;
        p.dst = dst;
        p.head = (int)head;
        p.nvec = (n - head) >> 4;
        p.tail = (int)((n - head) & 15);
        has = n > 0;
      }
      s_has[s][j] = has ? 1 : 0;
    }
    consumer_sync();
    // Compact list of each segment's non-empty pieces (consumer warp s).
    if (ct / 32 < nbatch) {
      const int s = ct / 32;
      const bool h0 = lane < P && s_has[s][lane];
      const bool h1 = lane + 32 < P && s_has[s][lane + 32];
      const unsigned m0 = __ballot_sync(kFull, h0);
      const unsigned m1 = __ballot_sync(kFull, h1);
      const unsigned below = (1u << lane) - 1u;
      if (h0) s_list[s][__popc(m0 & below)] = lane;
      if (h1) s_list[s][__popc(m0) + __popc(m1 & below)] = lane + 32;
      if (lane == 0) s_np[s] = __popc(m0) + __popc(m1);
    }
    consumer_sync();

    // This group's chunks of the batch: global chunk indices t = g mod kGroups.
    const int64_t tb = s_chbase[b0], te = s_chbase[b0 + nbatch];
    int64_t t = tb + (((int64_t)g - tb % kGroups) + kGroups) % kGroups;
    int sg = b0, q = 0;
#pragma unroll 1
    for (; t < te && live; t += kGroups) {
      while (s_chbase[sg + 1] <= t) {
        ++sg;
        q = 0;
      }
      const int stage = (int)(t % stages);
      const uint32_t ph = (uint32_t)((t / stages) & 1);
      const bool waited = mbar_wait(smem_u32(&s_full[stage]), ph, abort_flag);
      live = __all_sync(kFull, waited);
      if (!live) break;
      const uintptr_t c0 = s_seg_g0[sg] + (uintptr_t)(t - s_chbase[sg]) * kChunk;
      const uintptr_t G1 = s_seg_g1[sg];
      const uintptr_t c1 = c0 + kChunk < G1 ? c0 + kChunk : G1;   // bytes this chunk writes
      const int s = sg - b0;
      copy_chunk(s_piece[s], s_list[s], s_np[s], q, c0, c1, ring_base + stage * kStageStride,
                 gt, head_warp, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_empty[stage]));
    }
  }
  if (!live) return;

  // Bookkeeping, entries (i, j) spread over every consumer thread of the grid.
  const int64_t PP = (int64_t)P * P;
#pragma unroll 1
  for (int64_t e = (int64_t)b * kConsumers + ct; e < PP; e += (int64_t)nb * kConsumers) {
    const int i = (int)(e / P), j = (int)(e % P);
    int64_t sd = 0, rd = 0;
    for (int k = 0; k < j; ++k) sd += cnt[i * P + k];
    for (int k = 0; k < i; ++k) rd += cnt[k * P + j];
    a.sd[(int64_t)i * P + j] = sd;
    a.rc[(int64_t)j * P + i] = cnt[i * P + j];
    a.rd[(int64_t)j * P + i] = rd;
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

// Ring stages that fit beside a P x P count matrix: a multiple of kGroups
// (each stage then belongs to one consumer group), at most kMaxStages.
int stages_for(const A2avDeviceInfo& di, int P) {
  const int cnt_bytes = (P * P * 8 + 127) / 128 * 128;
  int s = (di.dyn_max - cnt_bytes) / kStageStride;
  s = s > kMaxStages ? kMaxStages : s;
  return s / kGroups * kGroups;
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
  a.stages = stages_for(di, a.P);
  if (a.stages < kGroups || a.stages % kGroups != 0 || blocks < 1)
    return cudaErrorInvalidConfiguration;
  const size_t dyn = (size_t)a.stages * kStageStride + (size_t)a.P * a.P * 8;
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
