// Tensor-core fused BMM -> TP ReduceScatter -> bias Add -> EP AllToAll for
// sm_103a: TMA loads into 128-byte-swizzled shared memory, tcgen05.mma with
// the fp32 accumulator in tensor memory, and an epilogue that writes each
// element straight to its final all-to-all destination.
//
// Dataflow (CANN guide "BatchMatMulReduceScatterAllToAll 原理、shape 约束与
// aclnn 两段式调用", 功能说明与计算流程): for source EP rank s and local
// expert e, the TP reduce-scatter sums x[s*tp+t][e] @ w[s*tp+t][e] over t.
// Here that sum is the contraction itself: the K loop of one output tile runs
// over t = 0..tp-1 (switching TMA descriptors at each shard boundary) and
// inside each shard over 64-wide K blocks, accumulating into the same TMEM
// accumulator, so the reduction is in fp32 in t order and temp1 / temp2 /
// temp3 never exist in memory.  The epilogue adds the sender's bias in fp32,
// rounds once and stores to y[j*tp+t] at block s*El+e, which is the
// all-to-all (chunk j of dim 1 to EP rank j, stacked by source rank then
// expert).
//
// Kernel shape: persistent, one 256-thread CTA per SM.
//   warp 0 (one lane)  TMA producer: per K block one 128x64 A box and four
//                      64x64 B boxes (B is the weight, N-contiguous) into a
//                      4-stage ring guarded by full/empty mbarriers.
//   warp 1 (one lane)  MMA issuer: tcgen05.mma.cta_group::1.kind::f16,
//                      M=128 N=256 K=16, four per K block; commits free the
//                      stage and, at the end of a tile, publish the
//                      accumulator.
//   warp 2             allocates / frees 512 TMEM columns: two 128x256 fp32
//                      accumulators, so the epilogue of one tile overlaps
//                      the K loop of the next.
//   warps 4..7         epilogue: tcgen05.ld 32 lanes x 32 columns at a time
//                      (warp w reads TMEM lanes 32*(w%4)...), bias, convert,
//                      16-byte stores.
// Every wait is bounded (about 4 s by %globaltimer); a wait that runs out
// records BRA_ERR_TIMEOUT in a device word, flags the CTA and every role
// leaves its loop, so the CTA still frees its tensor memory and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>
#include <memory>
#include <mutex>

#include "bra_internal.h"

namespace bra {

__device__ int32_t g_bra_fault_word = 0;

namespace {

#ifndef BRA_TC_STAGES
#define BRA_TC_STAGES 4
#endif
constexpr int BM = 128, BN = 256, BK = 64, STAGES = BRA_TC_STAGES;
constexpr int A_BYTES = BM * BK * 2;              // 16 KiB
constexpr int B_BOX_BYTES = 64 * BK * 2;          // one 64(N) x 64(K) box, 8 KiB
constexpr int B_BYTES = BN * BK * 2;              // 32 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;    // 48 KiB
constexpr int THREADS = 256;
constexpr int EPI_WARP0 = 4;
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
constexpr unsigned long long kWaitTimeoutNs = 4000000000ull;

struct TcParams {
  CUtensorMap tx[kChunkRanks];   // x_r: dims {Kp, ep*C, El}, box {64, 128, 1}
  CUtensorMap tw[kChunkRanks];   // w_r: dims {H, Kp, El},    box {64, 64, 1}
  const void* bias[kChunkRanks];
  void* y[kMaxRanks];
  int ep, tp, El, C, Kp, H, type, has_bias;
  int s0;                        // first source EP rank of this launch
  int nranks;                    // ranks of this launch (x / weight / bias)
  int rows;                      // ep * C
  int m_tiles, n_tiles, k_blocks, num_tiles;
  uint32_t idesc;                // tcgen05 instruction descriptor
  uint32_t b_lbo, b_sbo;         // B operand strides (bytes)
};

// ---------------------------------------------------------------------------
// PTX wrappers
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
// flagged by another role or the wait ran out (then this call flags it).
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
      atomicExch(&g_bra_fault_word, (int32_t)BRA_ERR_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ void spin_ns(unsigned long long ns) {
  const unsigned long long t0 = global_ns();
  while (global_ns() - t0 < ns) {
  }
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
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

// Tile index -> (local group, m tile, n tile).  Within a group the tiles
// are walked in super-rows of kGroupM m tiles: n tile by n tile, and inside
// each n tile down the super-row's m tiles.  CTAs running at the same time
// then share a few weight column bands and a few token row bands, and the
// next wave reuses the super-row's token rows from L2.
#ifndef BRA_TC_GROUP_M
#define BRA_TC_GROUP_M 16
#endif
constexpr int kGroupM = BRA_TC_GROUP_M;
struct TileCoord {
  int g, mt, nt;
};
__device__ __forceinline__ TileCoord tile_coord(const TcParams& p, int tile) {
  TileCoord c;
  const int per_group = p.m_tiles * p.n_tiles;
  c.g = tile / per_group;
  const int t = tile - c.g * per_group;
  if (kGroupM <= 0) {
    c.mt = t / p.n_tiles;
    c.nt = t - c.mt * p.n_tiles;
    return c;
  }
  const int span = kGroupM * p.n_tiles;          // tiles in one full super-row
  const int sr = t / span;
  const int first_m = sr * kGroupM;
  const int rows = min(kGroupM, p.m_tiles - first_m);
  const int u = t - sr * span;
  c.mt = first_m + u % rows;
  c.nt = u / rows;
  return c;
}

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

// ---------------------------------------------------------------------------
// Kernel
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(THREADS, 1) fused_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t smem_base = smem_u32(smem);
  uint8_t* bars = smem + STAGES * STAGE_BYTES;
  const uint32_t bar_base = smem_u32(bars);
  // barrier layout (8 bytes each): full[STAGES], empty[STAGES], tfull[2], tempty[2]
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 + a); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8 * (2 * STAGES + 4));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 8 * (2 * STAGES + 4) + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);   // one arrival per epilogue warp
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    for (int r = 0; r < p.nranks; ++r) {
      tma_prefetch_desc(&p.tx[r]);
      tma_prefetch_desc(&p.tw[r]);
    }
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const TileCoord tc = tile_coord(p, tile);
      const int sl = tc.g / p.El, e = tc.g % p.El;
      for (int t = 0; ok && t < p.tp; ++t) {
        const int r = sl * p.tp + t;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_expect_tx(fb, STAGE_BYTES);
          const uint32_t a_dst = smem_base + stage * STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          tma_load_3d(a_dst, &p.tx[r], fb, kb * BK, tc.mt * BM, e);
#pragma unroll
          for (int c = 0; c < BN / 64; ++c)
            tma_load_3d(b_dst + c * B_BOX_BYTES, &p.tw[r], fb, tc.nt * BN + c * 64, kb * BK, e);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    if (!ok) spin_ns(2000000ull);   // let copies already issued land
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      const int kk_total = p.tp * p.k_blocks;
      for (int kk = 0; kk < kk_total; ++kk) {
        if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_base + stage * STAGE_BYTES;
        const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          // A: K-major, 128-byte rows; K step of 16 elements = 32 bytes.
          const uint64_t ad = smem_desc_sw128(a_addr + k * 32, 16, 1024);
          // B: N-major boxes of 64(N) x 64(K); K step of 16 rows = 2048 bytes.
          const uint64_t bd = smem_desc_sw128(b_addr + k * 2048, p.b_lbo, p.b_sbo);
          tc_mma(d_tmem, ad, bd, p.idesc, (kk > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(empty_bar(stage));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit(tfull_bar(acc));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // Drain: wait until every MMA this thread issued has completed.
    if (!ok) spin_ns(2000000ull);
  } else if (warp >= EPI_WARP0) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;                      // TMEM lane quarter
    const int row_in_tile = q * 32 + lane;
    const int Hp = p.H / p.tp;
    const int Cp = p.type == 1 ? p.C / p.tp : 1;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      const TileCoord tc = tile_coord(p, tile);
      const int sl = tc.g / p.El, e = tc.g % p.El;
      const int s = p.s0 + sl;
      // The whole warp leaves together if any lane's wait gave up, so the
      // warp-wide tcgen05.ld below always runs on all 32 lanes.
      const bool waited = mbar_wait(tfull_bar(acc), acc_phase, abort_flag);
      if (!__all_sync(0xffffffffu, waited)) break;
      tc_fence_after();
      const int m = tc.mt * BM + row_in_tile;
      const bool row_ok = m < p.rows;
      const int j = row_ok ? m / p.C : 0;
      const int cm = row_ok ? m % p.C : 0;
      // yShardType 1: the row picks the TP destination and its row there.
      int t1 = 0;
      int64_t row1 = 0;
      if (p.type == 1) {
        t1 = cm / Cp;
        row1 = ((int64_t)(s * p.El + e) * Cp + (cm % Cp)) * p.H;
      }
      const uint32_t t_base = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(t_base + ch * 32, v);
        tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            const int n = tc.nt * BN + ch * 32 + g8 * 8;
            if (n < p.H) {
              int t;
              int64_t off, boff;
              if (p.type == 0) {
                t = n / Hp;
                const int h = n - t * Hp;
                off = ((int64_t)(s * p.El + e) * p.C + cm) * Hp + h;
                boff = (int64_t)e * Hp + h;
              } else {
                t = t1;
                off = row1 + n;
                boff = (int64_t)e * p.H + n;
              }
              float f[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) f[k] = __uint_as_float(v[g8 * 8 + k]);
              if (p.has_bias) {
                float b[8];
                Out<T>::bias8(static_cast<const uint8_t*>(p.bias[sl * p.tp + t]) +
                                  boff * Out<T>::kBiasBytes,
                              b);
#pragma unroll
                for (int k = 0; k < 8; ++k) f[k] += b[k];
              }
              uint4 o;
              o.x = Out<T>::pack(f[0], f[1]);
              o.y = Out<T>::pack(f[2], f[3]);
              o.z = Out<T>::pack(f[4], f[5]);
              o.w = Out<T>::pack(f[6], f[7]);
              T* yd = static_cast<T*>(p.y[j * p.tp + t]);
              *reinterpret_cast<uint4*>(yd + off) = o;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

bool encode_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t d0, uint64_t d1,
               uint64_t d2, uint32_t b0, uint32_t b1) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// tcgen05 instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B
// type (bits 7-9, 10-12: 0 fp16, 1 bf16), A K-major (bit 15 = 0), B N-major
// (bit 16 = 1), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
uint32_t make_idesc(bool bf16) {
  const uint32_t ab = bf16 ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | (0u << 15) | (1u << 16) |
         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

struct DeviceInfo {
  int sms = 0;
  bool attr_set = false;
};

}  // namespace

bool fused_tc_eligible(const FusedProblem& f) {
  if (f.Kp % 8 != 0 || f.H % 8 != 0) return false;
  if (f.type == 0 && (f.H / f.tp) % 8 != 0) return false;
  const int P = f.ep * f.tp;
  if (P > kMaxRanks) return false;
  auto al = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  for (int r = 0; r < P; ++r) {
    if (!al(f.x[r]) || !al(f.w[r]) || !al(f.y[r])) return false;
    if (f.bias && !al(f.bias[r])) return false;
  }
  return true;
}

cudaError_t launch_fused_tc(const FusedProblem& f, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static DeviceInfo info[64];
  int sms = 148;
  {
    std::lock_guard<std::mutex> lk(mu);
    DeviceInfo& di = info[dev & 63];
    if (!di.attr_set) {
      e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(fused_tc_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SMEM_BYTES);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(fused_tc_kernel<__nv_bfloat16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
      if (e != cudaSuccess) return e;
      di.attr_set = true;
    }
    sms = di.sms;
  }

  std::unique_ptr<TcParams> p(new TcParams);
  std::memset(p.get(), 0, sizeof(TcParams));
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
  p->rows = f.ep * f.C;
  p->m_tiles = (p->rows + BM - 1) / BM;
  p->n_tiles = (f.H + BN - 1) / BN;
  p->k_blocks = (f.Kp + BK - 1) / BK;
  const bool bf16 = f.dtype == BRA_BF16;
  p->idesc = make_idesc(bf16);
  p->b_lbo = B_BOX_BYTES;   // next 64-wide N group
  p->b_sbo = 1024;          // next 8 K rows
  const CUtensorMapDataType dt =
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int s_per_launch = kChunkRanks / f.tp > 0 ? kChunkRanks / f.tp : 1;
  for (int s0 = 0; s0 < f.ep; s0 += s_per_launch) {
    const int s1 = s0 + s_per_launch < f.ep ? s0 + s_per_launch : f.ep;
    p->s0 = s0;
    p->nranks = (s1 - s0) * f.tp;
    for (int r = 0; r < (s1 - s0) * f.tp; ++r) {
      const int gr = s0 * f.tp + r;
      if (!encode_3d(&p->tx[r], dt, f.x[gr], (uint64_t)f.Kp, (uint64_t)p->rows, (uint64_t)f.El,
                     BK, BM))
        return cudaErrorInvalidValue;
      if (!encode_3d(&p->tw[r], dt, f.w[gr], (uint64_t)f.H, (uint64_t)f.Kp, (uint64_t)f.El, 64,
                     BK))
        return cudaErrorInvalidValue;
      p->bias[r] = f.bias ? f.bias[gr] : nullptr;
    }
    p->num_tiles = (s1 - s0) * f.El * p->m_tiles * p->n_tiles;
    const int grid = p->num_tiles < sms ? p->num_tiles : sms;
    if (bf16)
      fused_tc_kernel<__nv_bfloat16><<<grid, THREADS, SMEM_BYTES, st>>>(*p);
    else
      fused_tc_kernel<__half><<<grid, THREADS, SMEM_BYTES, st>>>(*p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t read_fault_word(int32_t* code, int clear) {
  cudaError_t e = cudaMemcpyFromSymbol(code, g_bra_fault_word, sizeof(int32_t));
  if (e != cudaSuccess) return e;
  if (clear) {
    const int32_t z = 0;
    e = cudaMemcpyToSymbol(g_bra_fault_word, &z, sizeof(int32_t));
  }
  return e;
}

}  // namespace bra
