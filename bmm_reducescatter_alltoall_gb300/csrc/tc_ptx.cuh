// Inline-PTX building blocks shared by the sm_103a tensor-core fused kernels
// (fused_tc.cu: one CTA per tile; fused_tc2.cu: a CTA pair per tile).
//
// mbarrier, TMA (cp.async.bulk.tensor), tcgen05 (alloc / mma / commit / ld),
// the 128-byte-swizzle shared-memory matrix descriptor, cluster helpers, the
// tile raster and the epilogue that turns one accumulator row into stores at
// the all-to-all destinations.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <mutex>

#include "bra_internal.h"

namespace bra {
namespace tc {

constexpr unsigned long long kWaitTimeoutNs = 4000000000ull;

// Kernel parameters of both tensor-core kernels (passed as __grid_constant__).
struct TcParams {
  CUtensorMap tx[kChunkRanks];   // x_r: dims {Kp, ep*C, El}
  CUtensorMap tw[kChunkRanks];   // w_r: dims {H, Kp, El}
  const void* bias[kChunkRanks];
  void* y[kMaxRanks];
  int ep, tp, El, C, Kp, H, type, has_bias;
  int s0;                        // first source EP rank of this launch
  int nranks;                    // ranks of this launch (x / weight / bias)
  int rows;                      // ep * C
  int m_tiles, n_tiles, k_blocks, num_tiles;
  uint32_t idesc;                // tcgen05 instruction descriptor
  uint32_t b_lbo, b_sbo;         // B operand strides (bytes), N-major weight
  int b_kmajor;                  // weight stored transposed: B is K-major
  int y_elem;                    // output rows / pointers or bias not 16-byte aligned:
                                 // the element-wise epilogue (tcu_epilogue.cuh)
  int32_t* status;               // per-call timeout word (optional)
};

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
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
// Arrive on a barrier given by its shared::cluster address (any CTA of the
// cluster), with release semantics at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
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
// and records BRA_ERR_TIMEOUT in *fault_word).  mbar_wait below checks the
// phase inline first and only calls this slow path when it has to wait.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                                   volatile int* abort_flag, int32_t* fault_word) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int k = 0; k < 64; ++k)
      if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitTimeoutNs) {
      *abort_flag = 1;
      atomicExch(fault_word, (int32_t)BRA_ERR_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* fault_word) {
  return mbar_try(bar, parity) || mbar_wait_slow(bar, parity, abort_flag, fault_word);
}
__device__ __forceinline__ void spin_ns(unsigned long long ns) {
  const unsigned long long t0 = global_ns();
  while (global_ns() - t0 < ns) {
  }
}

// ---------------------------------------------------------------------------
// cluster
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared variable in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
// Whole-cluster barrier; every thread of every CTA, converged warps.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Load into this CTA's shared memory, completing on a barrier that may live
// in either CTA of the pair (cluster_bar is a shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t cluster_bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// The same, multicast to the CTAs of `cta_mask` (same shared-memory offset in
// each); each destination's bytes complete on the barrier at cluster_bar's
// offset in the leader of the destination's own CTA pair.
__device__ __forceinline__ void tma_load_3d_pair_mc(uint32_t dst, const CUtensorMap* map,
                                                    uint32_t cluster_bar, int c0, int c1, int c2,
                                                    uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2),
      "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// With CG == 2 one warp of each CTA of the pair issues these together; the
// pair gets the same column range in both CTAs.
template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_relinquish() {
  if constexpr (CG == 1)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// D (TMEM) [+]= A (smem) x B (smem), kind::f16 (fp16 or bf16 in, fp32 acc).
template <int CG>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  if constexpr (CG == 1)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// Pair form: arrive on the barrier at the same shared offset in every CTA
// of `cta_mask`.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2), version
// 1: start address, leading and stride byte offsets in 16-byte units.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// tcgen05 instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B
// type (bits 7-9, 10-12: 0 fp16, 1 bf16), A K-major (bit 15 = 0), B N-major
// (bit 16 = 1) or K-major (bit 16 = 0, transposed weight), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
inline uint32_t make_idesc(bool bf16, int M, int N, bool b_kmajor = false) {
  const uint32_t ab = bf16 ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | (0u << 15) | ((b_kmajor ? 0u : 1u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Operand descriptors of one CTA's ring, built once: the descriptor of any
// stage / K step is the base descriptor plus the byte offset in 16-byte
// units (the 14-bit start-address field; shared memory is below 256 KiB, so
// the add never carries out of it).  A is K-major (K step of 16 elements =
// 32 bytes); B is N-major boxes of 64(N) x 64(K) (K step = 16 rows = 2048
// bytes) or, for a transposed weight, K-major (32 bytes).
struct RingDescs {
  uint64_t a0, b0;        // stage 0, K step 0
  uint32_t b_kstep;       // B K step, 16-byte units
};
__device__ __forceinline__ RingDescs ring_descs(const TcParams& p, uint32_t a_addr0,
                                                uint32_t b_addr0) {
  RingDescs d;
  d.a0 = smem_desc_sw128(a_addr0, 16, 1024);
  d.b0 = p.b_kmajor ? smem_desc_sw128(b_addr0, 16, 1024)
                    : smem_desc_sw128(b_addr0, p.b_lbo, p.b_sbo);
  d.b_kstep = p.b_kmajor ? 2u : 128u;
  return d;
}

// ---------------------------------------------------------------------------
// Tile raster: within a group the tiles are walked in super-rows of kGroupM
// m tiles: n tile by n tile, and inside each n tile down the super-row's m
// tiles.  CTAs running at the same time then share a few weight column bands
// and a few token row bands, and the next wave reuses the super-row's token
// rows from L2.
// ---------------------------------------------------------------------------
struct TileCoord {
  int g, mt, nt;
};
__device__ __forceinline__ TileCoord tile_coord(int tile, int m_tiles, int n_tiles, int group_m) {
  TileCoord c;
  const int per_group = m_tiles * n_tiles;
  c.g = tile / per_group;
  const int t = tile - c.g * per_group;
  if (group_m <= 0) {
    c.mt = t / n_tiles;
    c.nt = t - c.mt * n_tiles;
    return c;
  }
  const int span = group_m * n_tiles;
  const int sr = t / span;
  const int first_m = sr * group_m;
  const int rows = min(group_m, m_tiles - first_m);
  const int u = t - sr * span;
  c.mt = first_m + u % rows;
  c.nt = u / rows;
  return c;
}

// ---------------------------------------------------------------------------
// Epilogue
// ---------------------------------------------------------------------------
template <typename T>
struct Out;
template <>
struct Out<__half> {
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  // 8 bias values (fp16) starting at p.
  static __device__ __forceinline__ void bias8(const void* p, float (&b)[8]) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __half22float2(h[k]);
      b[2 * k] = f.x;
      b[2 * k + 1] = f.y;
    }
  }
  static constexpr int kBiasBytes = 2;
};
template <>
struct Out<__nv_bfloat16> {
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  // 8 bias values (fp32) starting at p.
  static __device__ __forceinline__ void bias8(const void* p, float (&b)[8]) {
    const float4 u = __ldg(reinterpret_cast<const float4*>(p));
    const float4 v = __ldg(reinterpret_cast<const float4*>(p) + 1);
    b[0] = u.x; b[1] = u.y; b[2] = u.z; b[3] = u.w;
    b[4] = v.x; b[5] = v.y; b[6] = v.z; b[7] = v.w;
  }
  static constexpr int kBiasBytes = 4;
};

// Shared-memory staging per epilogue warp: 32 rows x 64 columns of the
// output dtype (128 bytes) with rows 144 bytes apart, so the row-per-lane
// writes and the row-segment reads are both free of bank conflicts.
constexpr int kEpiRowStride = 144;
constexpr int kEpiBiasBytes = 512 * 4;                // bias of up to 512 columns, fp32
constexpr int kEpiStageBytes = 32 * kEpiRowStride + kEpiBiasBytes;   // per warp

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 lds128e(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// The epilogue of one warp (epilogue_rows below: epilogue_bias, then
// epilogue_body) drains its 32 TMEM lanes (accumulator rows row0 .. row0+31
// of Z_{s,e}, the global row index in ep*C) of a BN-column accumulator,
// columns n0 .. n0+BN-1, 64 columns at a time:
//   1. lane l holds row row0+l: tcgen05.ld two 32-column slices, add the
//      sender's bias in fp32, round once, write the 128-byte row segment to
//      the warp's staging tile;
//   2. the warp stores the staging tile row segment by row segment: lanes
//      8r'..8r'+7 write the 8 x 16 bytes of one row, 4 rows per instruction,
//      each to its all-to-all destination
//        yShardType 0: y[j*tp + n/Hp][s*El+e, m%C, n%Hp]
//        yShardType 1: y[j*tp + (m%C)/Cp][s*El+e, (m%C)%Cp, n]   (j = m / C).
// Every lane runs the warp-wide tcgen05.ld; stores are masked per row and
// per 8 columns (H is a multiple of 8).
// Bias staging of the tile (step 0 of the epilogue, which the caller may run
// before the accumulator is ready: it depends on the tile's coordinates
// only).  When the bias depends on the column only -- always for
// yShardType 0, and for yShardType 1 when the warp's 32 rows share a TP rank
// (row 0 of the warp is valid whenever any is) -- the warp stages the tile's
// BN bias values (fp32) once in its staging tile and every row reads them
// by broadcast; returns whether it did (warp-uniform).
template <typename T, int BN>
__device__ __forceinline__ bool epilogue_bias(const TcParams& p, int row0, int sl, int e, int n0,
                                              uint32_t stage, int lane) {
  static_assert(BN * 4 <= kEpiBiasBytes, "bias staging");
  const int Hp = p.H / p.tp;
  const int Cp = p.type == 1 ? p.C / p.tp : 1;
  const int m_own = row0 + lane;
  const bool own_ok = m_own < p.rows;
  const int t_own = (own_ok && p.type == 1) ? (m_own % p.C) / Cp : 0;
  const int t_first = __shfl_sync(0xffffffffu, t_own, 0);
  const uint32_t bias_stage = stage + 32 * kEpiRowStride;
  const bool bias_staged =
      p.has_bias && (p.type == 0 || __all_sync(0xffffffffu, !own_ok || t_own == t_first));
  if (bias_staged) {
    for (int g = lane; g < BN / 8; g += 32) {
      const int n = n0 + g * 8;
      float b[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (n < p.H) {
        if (p.type == 0) {
          const int t = n / Hp;
          Out<T>::bias8(static_cast<const uint8_t*>(p.bias[sl * p.tp + t]) +
                            ((int64_t)e * Hp + (n - t * Hp)) * Out<T>::kBiasBytes,
                        b);
        } else {
          Out<T>::bias8(static_cast<const uint8_t*>(p.bias[sl * p.tp + t_first]) +
                            ((int64_t)e * p.H + n) * Out<T>::kBiasBytes,
                        b);
        }
      }
      sts128(bias_stage + g * 32, make_uint4(__float_as_uint(b[0]), __float_as_uint(b[1]),
                                             __float_as_uint(b[2]), __float_as_uint(b[3])));
      sts128(bias_stage + g * 32 + 16, make_uint4(__float_as_uint(b[4]), __float_as_uint(b[5]),
                                                  __float_as_uint(b[6]), __float_as_uint(b[7])));
    }
  }
  __syncwarp();
  return bias_staged;
}

// The rest of the epilogue, once the accumulator is ready (bias_staged: what
// epilogue_bias returned for this tile).  The next 64 columns' TMEM loads are
// issued as soon as a chunk is staged, so they land while the chunk's stores
// go out.  tmem_done() runs on every lane right after the last TMEM load has
// landed: the accumulator may be handed back there, before the last chunk's
// conversion and stores.
template <typename T, int BN, typename TmemDone>
__device__ __forceinline__ void epilogue_body(const TcParams& p, uint32_t t_base, int row0, int sl,
                                              int e, int n0, uint32_t stage, int lane,
                                              bool bias_staged, TmemDone&& tmem_done) {
  const int s = p.s0 + sl;
  const int Hp = p.H / p.tp;
  const int Cp = p.type == 1 ? p.C / p.tp : 1;
  // this lane's own row (phase 1)
  const int m_own = row0 + lane;
  const bool own_ok = m_own < p.rows;
  const int t_own = (own_ok && p.type == 1) ? (m_own % p.C) / Cp : 0;
  const uint32_t bias_stage = stage + 32 * kEpiRowStride;
  // the 8 rows this lane stores (phase 2): r = 4q + lane/8
  const int kc = lane & 7;
  int64_t rbase[8];
  int rdest[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int m = row0 + 4 * q + (lane >> 3);
    if (m < p.rows) {
      const int j = m / p.C, cm = m % p.C;
      if (p.type == 0) {
        rbase[q] = ((int64_t)(s * p.El + e) * p.C + cm) * Hp;
        rdest[q] = j * p.tp;
      } else {
        rbase[q] = ((int64_t)(s * p.El + e) * Cp + (cm % Cp)) * p.H;
        rdest[q] = j * p.tp + cm / Cp;
      }
    } else {
      rdest[q] = -1;
    }
  }
  const uint32_t my_row = stage + (uint32_t)lane * kEpiRowStride;
  uint32_t v[64];
  tmem_ld32(t_base, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
  tmem_ld32(t_base + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
#pragma unroll 1
  for (int ch = 0; ch < BN / 64; ++ch) {
    tmem_ld_wait();
    if (ch + 1 == BN / 64) tmem_done();
    // phase 1: bias, convert, stage the row segment.  Loads are issued in
    // batches ahead of their use (shared-memory accesses here are ordered
    // asm statements, so a load placed after a store would wait for it).
    if (bias_staged) {
#pragma unroll
      for (int bq = 0; bq < 4; ++bq) {          // 16 columns per batch
        uint4 b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          b[i] = lds128e(bias_stage + (uint32_t)(ch * 64 + bq * 16 + i * 4) * 4);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t* w = &v[bq * 16 + i * 4];
          w[0] = __float_as_uint(__uint_as_float(w[0]) + __uint_as_float(b[i].x));
          w[1] = __float_as_uint(__uint_as_float(w[1]) + __uint_as_float(b[i].y));
          w[2] = __float_as_uint(__uint_as_float(w[2]) + __uint_as_float(b[i].z));
          w[3] = __float_as_uint(__uint_as_float(w[3]) + __uint_as_float(b[i].w));
        }
      }
    } else if (p.has_bias && own_ok) {
      // yShardType 1, rows of several TP ranks: each row its own bias row.
#pragma unroll
      for (int g8 = 0; g8 < 8; ++g8) {
        const int n = n0 + ch * 64 + g8 * 8;
        if (n < p.H) {
          float b[8];
          Out<T>::bias8(static_cast<const uint8_t*>(p.bias[sl * p.tp + t_own]) +
                            ((int64_t)e * p.H + n) * Out<T>::kBiasBytes,
                        b);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            v[g8 * 8 + k] = __float_as_uint(__uint_as_float(v[g8 * 8 + k]) + b[k]);
        }
      }
    }
    uint32_t o[32];
#pragma unroll
    for (int k = 0; k < 32; ++k)
      o[k] = Out<T>::pack(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
#pragma unroll
    for (int g8 = 0; g8 < 8; ++g8)
      sts128(my_row + g8 * 16, make_uint4(o[4 * g8], o[4 * g8 + 1], o[4 * g8 + 2], o[4 * g8 + 3]));
    // the next chunk's accumulator columns, into the registers just consumed
    if (ch + 1 < BN / 64) {
      tmem_ld32(t_base + (ch + 1) * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(t_base + (ch + 1) * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
    }
    __syncwarp();
    // phase 2: row segments to their destinations, all eight loaded first
    const int n = n0 + ch * 64 + kc * 8;
    if (n < p.H) {
      const int t0 = p.type == 0 ? n / Hp : 0;
      const int h0 = n - t0 * Hp;
      uint4 val[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        val[q] = lds128e(stage + (uint32_t)(4 * q + (lane >> 3)) * kEpiRowStride + kc * 16);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (rdest[q] < 0) continue;
        int d;
        int64_t off;
        if (p.type == 0) {
          d = rdest[q] + t0;
          off = rbase[q] + h0;
        } else {
          d = rdest[q];
          off = rbase[q] + n;
        }
        T* yd = static_cast<T*>(p.y[d]);
        *reinterpret_cast<uint4*>(yd + off) = val[q];
      }
    }
    __syncwarp();
  }
}

// The whole epilogue of one warp (bias staging, then the body).
template <typename T, int BN>
__device__ __forceinline__ void epilogue_rows(const TcParams& p, uint32_t t_base, int row0, int sl,
                                              int e, int n0, uint32_t stage, int lane) {
  const bool bias_staged = epilogue_bias<T, BN>(p, row0, sl, e, n0, stage, lane);
  epilogue_body<T, BN>(p, t_base, row0, sl, e, n0, stage, lane, bias_staged, [] {});
}

// ---------------------------------------------------------------------------
// Host helpers
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 3-D 16-bit tensor {d0 (contiguous), d1, d2} whose rows are `pitch`
// elements apart (pitch >= d0), box {b0, b1, 1}, 128-byte swizzle, zero fill
// outside the tensor (including columns d0 .. pitch-1).
inline bool encode_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t d0,
                      uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1, uint64_t pitch) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {pitch * 2, pitch * d1 * 2};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Fill the fields of TcParams common to every launch of one problem.
inline void fill_common(TcParams* p, const FusedProblem& f, int bm, int bn, int bk) {
  const int P = f.ep * f.tp;
  for (int d = 0; d < P; ++d) p->y[d] = f.y[d];
  p->ep = f.ep;
  p->tp = f.tp;
  p->El = f.El;
  p->C = f.C;
  p->Kp = f.Kp;
  p->H = f.H;
  p->type = f.type;
  p->has_bias = f.bias != nullptr;
  p->b_kmajor = f.wt;
  p->status = f.status;
  p->rows = f.ep * f.C;
  // 16-byte vector stores need 16-byte output rows and pointers, and the
  // vector bias loads 16-byte bias rows and pointers.
  {
    const int Hp = f.H / f.tp;
    bool vec = (f.type == 1 ? f.H : Hp) % 8 == 0;
    auto al = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    for (int d = 0; vec && d < P; ++d) vec = al(f.y[d]) && (!f.bias || al(f.bias[d]));
    p->y_elem = vec ? 0 : 1;
  }
  p->m_tiles = (p->rows + bm - 1) / bm;
  p->n_tiles = (f.H + bn - 1) / bn;
  p->k_blocks = (f.Kp + bk - 1) / bk;
}

// Descriptors and bias pointers of the source ranks [s0, s1).  The weight
// box is 64 columns x bk rows for the N-major weight, or bk x b_rows_t
// (K x N) for the transposed (K-major) weight.
inline bool fill_chunk(TcParams* p, const FusedProblem& f, int s0, int s1, uint32_t a_rows,
                       uint32_t b_cols, int bk, uint32_t b_rows_t) {
  const CUtensorMapDataType dt =
      f.dtype == BRA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  p->s0 = s0;
  p->nranks = (s1 - s0) * f.tp;
  for (int r = 0; r < p->nranks; ++r) {
    const int gr = s0 * f.tp + r;
    if (!encode_3d(&p->tx[r], dt, f.x[gr], (uint64_t)f.Kp, (uint64_t)p->rows, (uint64_t)f.El,
                   (uint32_t)bk, a_rows, (uint64_t)f.xp))
      return false;
    const bool ok = f.wt ? encode_3d(&p->tw[r], dt, f.w[gr], (uint64_t)f.Kp, (uint64_t)f.H,
                                     (uint64_t)f.El, (uint32_t)bk, b_rows_t, (uint64_t)f.wp)
                         : encode_3d(&p->tw[r], dt, f.w[gr], (uint64_t)f.H, (uint64_t)f.Kp,
                                     (uint64_t)f.El, b_cols, (uint32_t)bk, (uint64_t)f.wp);
    if (!ok) return false;
    p->bias[r] = f.bias ? f.bias[gr] : nullptr;
  }
  return true;
}

}  // namespace tc
}  // namespace bra
