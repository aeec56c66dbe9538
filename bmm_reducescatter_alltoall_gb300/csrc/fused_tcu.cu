// Tensor-core fused BMM -> TP ReduceScatter -> bias Add -> EP AllToAll for
// shapes whose rows are not 16-byte aligned (M/tp, H or H/tp not a multiple
// of 8 elements, e.g. the 8-rank example of the CANN guide "BatchMatMul
// ReduceScatterAllToAll 原理、shape 约束与 aclnn 两段式调用", 完整调用示例,
// with M/tp = 6 and H = 4), where TMA cannot describe the operands.
//
// The dataflow is that of fused_tc.cu (功能说明与计算流程): for source EP
// rank s and local expert e the K loop of a 128 x 256 output tile runs over
// the tp shards t = 0..tp-1 and, inside each, over 64-wide K blocks, so the
// TP reduce-scatter is the fp32 accumulation itself, in t order; the
// epilogue adds the sender's bias, rounds once and stores each element at its
// all-to-all destination.  What differs is how operands reach shared memory:
//   warps 5..12  producers: every 16-byte chunk of a stage (128 x 64 A and
//                64 x 256 B elements, laid out exactly as a 128-byte-swizzle
//                TMA box would be) is read with the aligned 16-byte loads that
//                cover it, funnel-shifted into place and masked past the end
//                of a row, written with st.shared, made visible to the tensor
//                core with fence.proxy.async, and published on the stage's
//                full barrier (one arrival per producer warp).  A loaded
//                16-byte granule always holds a byte of the operand, so no
//                load leaves a page the operand does not touch.
//   warp 4       allocates 512 TMEM columns (two 128 x 256 fp32
//                accumulators); its lane 0 issues tcgen05.mma (M=128, N=256,
//                K=16) and commits stages and accumulators.
//   warps 0..3   epilogue (tcu_epilogue.cuh): tcgen05.ld of the warp's TMEM
//                lane quarter, bias, one rounding; each row segment staged
//                in shared memory shifted to its destination's 16-byte phase
//                and written with aligned vector stores (partial end chunks
//                and segments that straddle a TP rank's chunk piecewise), so
//                rows of any alignment are fine.
// Every wait is bounded (about 4 s); a wait that runs out records
// BRA_ERR_TIMEOUT in a device word and every role leaves its loop.
#include <cstring>
#include <memory>
#include <mutex>

#include "tcu_epilogue.cuh"

namespace bra {

__device__ int32_t g_bra_fault_word3 = 0;

namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int kGroupM = 16;
constexpr int A_BYTES = BM * BK * 2;              // 16 KiB
constexpr int B_BOX_BYTES = 64 * BK * 2;          // 64(N) x 64(K), 8 KiB
constexpr int B_BYTES = BN * BK * 2;              // 32 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;    // 48 KiB
constexpr int A_CHUNKS = A_BYTES / 16, B_CHUNKS = B_BYTES / 16;
#ifndef BRA_TCU_PROD_WARPS
#define BRA_TCU_PROD_WARPS 7
#endif
constexpr int EPI_WARPS = 4, MMA_WARP = 4, PROD_WARP0 = 5, PROD_WARPS = BRA_TCU_PROD_WARPS;
constexpr int THREADS = (PROD_WARP0 + PROD_WARPS) * 32;
constexpr int PROD_THREADS = PROD_WARPS * 32;
constexpr int CHUNKS_PER_THREAD = (A_CHUNKS + B_CHUNKS + PROD_THREADS - 1) / PROD_THREADS;
// Chunks whose loads are in flight together (13 warps leave 128 registers a
// thread: an SM sub-partition holds four of them).  Four spill a few bytes
// and still beat two and three, since throughput is set by the loads in
// flight.
#ifndef BRA_TCU_BATCH
#define BRA_TCU_BATCH 7
#endif
constexpr int BATCH = BRA_TCU_BATCH;
static_assert(CHUNKS_PER_THREAD % BATCH == 0, "batches");
constexpr int ALL_CHUNKS = A_CHUNKS + B_CHUNKS;
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + EPI_WARPS * kUStageBytes + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct UParams {
  const void* x[kChunkRanks];
  const void* w[kChunkRanks];
  const void* bias[kChunkRanks];
  void* y[kMaxRanks];
  int ep, tp, El, C, Kp, H, type, has_bias;
  int s0, rows, m_tiles, n_tiles, k_blocks, num_tiles;
  int b_kmajor;
  uint32_t idesc;
  int32_t* status;   // per-call timeout word (optional)
};

__device__ __forceinline__ uint4 ldg128(uintptr_t a) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(a));
  return v;
}

// The 16 bytes starting `delta` (even) bytes into the 32 bytes (a, b).
__device__ __forceinline__ uint4 realign_rt(const uint4& a, const uint4& b, uint32_t delta) {
  const bool two = (delta & 8u) != 0, one = (delta & 4u) != 0;
  const uint32_t r = (delta & 3u) * 8u;
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

// Keep the first n (0..8) 16-bit elements of v, zero the rest.
__device__ __forceinline__ uint4 keep_elems(uint4 v, int n) {
  auto w = [n](uint32_t x, int i) -> uint32_t {
    return n >= 2 * i + 2 ? x : (n == 2 * i + 1 ? (x & 0xFFFFu) : 0u);
  };
  return make_uint4(w(v.x, 0), w(v.y, 1), w(v.z, 2), w(v.w, 3));
}

// One 16-byte chunk of eight consecutive elements of a row: `row` is the
// address of element 0 of the row, the chunk starts at element k and the row
// holds `len` elements (nothing when k >= len).  Only the aligned granules
// that hold one of the chunk's valid bytes are read.
struct ChunkLoad {
  uint4 a, b;
  uint32_t delta;
  int n;
};
__device__ __forceinline__ ChunkLoad chunk_issue(uintptr_t row, int k, int len, bool row_ok) {
  ChunkLoad c;
  c.n = row_ok ? min(max(len - k, 0), 8) : 0;
  c.a = make_uint4(0, 0, 0, 0);
  c.b = c.a;
  c.delta = 0;
  if (c.n > 0) {
    const uintptr_t addr = row + (uintptr_t)k * 2;
    const uintptr_t a0 = addr & ~(uintptr_t)15;
    c.delta = (uint32_t)(addr - a0);
    c.a = ldg128(a0);
    if (c.delta + 2u * (uint32_t)c.n > 16u) c.b = ldg128(a0 + 16);
  }
  return c;
}
__device__ __forceinline__ uint4 chunk_value(const ChunkLoad& c) {
  if (c.n == 0) return make_uint4(0, 0, 0, 0);
  uint4 v = c.delta ? realign_rt(c.a, c.b, c.delta) : c.a;
  return c.n < 8 ? keep_elems(v, c.n) : v;
}

template <typename T>
__global__ void __launch_bounds__(THREADS, 1) fused_tcu_kernel(const __grid_constant__ UParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t smem_base = smem_u32(smem);
  uint8_t* bars = smem + STAGES * STAGE_BYTES;
  const uint32_t bar_base = smem_u32(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 + a); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8 * (2 * STAGES + 4));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 8 * (2 * STAGES + 4) + 8);
  int32_t* fault = &g_bra_fault_word3;
  uint8_t* epi_smem = bars + BAR_BYTES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), PROD_WARPS);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), EPI_WARPS);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == MMA_WARP) {
    tmem_alloc<1>(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp >= PROD_WARP0) {
    // ---------------- producers ----------------
    const int ptid = threadIdx.x - PROD_WARP0 * 32;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const TileCoord tc = tile_coord(tile, p.m_tiles, p.n_tiles, kGroupM);
      const int sl = tc.g / p.El, e = tc.g % p.El;
      for (int t = 0; ok && t < p.tp; ++t) {
        const int r = sl * p.tp + t;
        const uintptr_t xb = reinterpret_cast<uintptr_t>(p.x[r]) +
                             (uintptr_t)((int64_t)e * p.rows * p.Kp * 2);
        const uintptr_t wb = reinterpret_cast<uintptr_t>(p.w[r]) +
                             (uintptr_t)((int64_t)e * p.Kp * p.H * 2);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          // The warp leaves together if any lane's wait gave up.
          const bool freed = mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, fault);
          if (!__all_sync(0xffffffffu, freed)) {
            ok = false;
            break;
          }
          const uint32_t a_dst = smem_base + stage * STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          const int k0 = kb * BK;
#pragma unroll
          for (int bt = 0; bt < CHUNKS_PER_THREAD / BATCH; ++bt) {
            ChunkLoad ld[BATCH];
            uint32_t dst[BATCH];
#pragma unroll
            for (int i = 0; i < BATCH; ++i) {
              const int id = ptid + (bt * BATCH + i) * PROD_THREADS;
              if (id >= ALL_CHUNKS) {
                ld[i].n = 0;
                dst[i] = 0;
              } else if (id < A_CHUNKS) {
                // A: token row m, K elements k0 + 8 kc ..
                const int rr = id >> 3, kc = id & 7;
                const int m = tc.mt * BM + rr;
                ld[i] = chunk_issue(xb + (uintptr_t)((int64_t)m * p.Kp * 2), k0 + kc * 8, p.Kp,
                                    m < p.rows);
                dst[i] = a_dst + rr * 128 + ((kc ^ (rr & 7)) << 4);
              } else if (!p.b_kmajor) {
                // B, weight (Kp, H): K row kr, N elements 8 cc .. of the tile
                const int b = id - A_CHUNKS, kr = b >> 5, cc = b & 31;
                const int k = k0 + kr;
                ld[i] = chunk_issue(wb + (uintptr_t)((int64_t)k * p.H * 2), tc.nt * BN + cc * 8,
                                    p.H, k < p.Kp);
                dst[i] = b_dst + (cc >> 3) * B_BOX_BYTES + kr * 128 + (((cc & 7) ^ (kr & 7)) << 4);
              } else {
                // B, transposed weight (H, Kp): N row n, K elements k0 + 8 kc ..
                const int b = id - A_CHUNKS, nr = b >> 3, kc = b & 7;
                const int n = tc.nt * BN + nr;
                ld[i] = chunk_issue(wb + (uintptr_t)((int64_t)n * p.Kp * 2), k0 + kc * 8, p.Kp,
                                    n < p.H);
                dst[i] = b_dst + nr * 128 + ((kc ^ (nr & 7)) << 4);
              }
            }
#pragma unroll
            for (int i = 0; i < BATCH; ++i)
              if (ptid + (bt * BATCH + i) * PROD_THREADS < ALL_CHUNKS)
                sts128(dst[i], chunk_value(ld[i]));
          }
          // generic-proxy writes -> visible to the tensor core, then publish
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(full_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      // Descriptors of stage 0, K step 0 (as the one-CTA TMA kernel builds them):
      // A K-major; B N-major boxes of 64 x 64 or, transposed, K-major.
      const uint64_t a0 = smem_desc_sw128(smem_base, 16, 1024);
      const uint64_t b0 = p.b_kmajor ? smem_desc_sw128(smem_base + A_BYTES, 16, 1024)
                                     : smem_desc_sw128(smem_base + A_BYTES, B_BOX_BYTES, 1024);
      const uint32_t b_kstep = p.b_kmajor ? 2u : 128u;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, fault)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        const int kk_total = p.tp * p.k_blocks;
        for (int kk = 0; kk < kk_total; ++kk) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, fault)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t so = (uint64_t)((stage * STAGE_BYTES) >> 4);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma<1>(d_tmem, a0 + so + 2 * k, b0 + so + b_kstep * k, p.idesc,
                      (kk > 0 || k > 0) ? 1u : 0u);
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
      if (!ok) spin_ns(2000000ull);   // let MMAs already issued complete
    }
  } else {
    // ---------------- epilogue (warps 0..3 = TMEM lane quarters) ----------------
    const int q = warp;
    uint8_t* stg = epi_smem + q * kUStageBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      const TileCoord tc = tile_coord(tile, p.m_tiles, p.n_tiles, kGroupM);
      const int sl = tc.g / p.El, e = tc.g % p.El;
      const bool waited = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, fault);
      if (!__all_sync(0xffffffffu, waited)) break;
      tc_fence_after();
      const uint32_t t_base = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      epilogue_rows_u<T, false>(p, t_base, tc.mt * BM + q * 32, sl, e, tc.nt * BN, stg, lane);
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
  if (threadIdx.x == 0 && p.status && *abort_flag) atomicExch(p.status, (int32_t)BRA_ERR_TIMEOUT);
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc<1>(tmem_base, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_fused_tcu(const FusedProblem& f, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static bool attr_set[64] = {};
  static int sms_of[64] = {};
  int sms = 148;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!attr_set[dev & 63]) {
      e = cudaDeviceGetAttribute(&sms_of[dev & 63], cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(fused_tcu_kernel<__half>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(fused_tcu_kernel<__nv_bfloat16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
      if (e != cudaSuccess) return e;
      attr_set[dev & 63] = true;
    }
    sms = sms_of[dev & 63];
  }
  std::unique_ptr<UParams> p(new UParams);
  std::memset(p.get(), 0, sizeof(UParams));
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
  p->status = f.status;
  p->b_kmajor = f.wt;
  p->rows = f.ep * f.C;
  p->m_tiles = (p->rows + BM - 1) / BM;
  p->n_tiles = (f.H + BN - 1) / BN;
  p->k_blocks = (f.Kp + BK - 1) / BK;
  p->idesc = make_idesc(f.dtype == BRA_BF16, BM, BN, f.wt != 0);
  const int s_per_launch = kChunkRanks / f.tp > 0 ? kChunkRanks / f.tp : 1;
  for (int s0 = 0; s0 < f.ep; s0 += s_per_launch) {
    const int s1 = s0 + s_per_launch < f.ep ? s0 + s_per_launch : f.ep;
    p->s0 = s0;
    for (int r = 0; r < (s1 - s0) * f.tp; ++r) {
      const int gr = s0 * f.tp + r;
      p->x[r] = f.x[gr];
      p->w[r] = f.w[gr];
      p->bias[r] = f.bias ? f.bias[gr] : nullptr;
    }
    p->num_tiles = (s1 - s0) * f.El * p->m_tiles * p->n_tiles;
    const int grid = p->num_tiles < sms ? p->num_tiles : sms;
    if (f.dtype == BRA_BF16)
      fused_tcu_kernel<__nv_bfloat16><<<grid, THREADS, SMEM_BYTES, st>>>(*p);
    else
      fused_tcu_kernel<__half><<<grid, THREADS, SMEM_BYTES, st>>>(*p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

bool fused_tcu_eligible(const FusedProblem& f) {
  // Element-aligned operands (2 bytes; bias 2 or 4) and at most kMaxRanks ranks.
  const int P = f.ep * f.tp;
  if (P > kMaxRanks) return false;
  const uintptr_t bias_align = f.dtype == BRA_BF16 ? 3u : 1u;
  for (int r = 0; r < P; ++r) {
    if ((reinterpret_cast<uintptr_t>(f.x[r]) | reinterpret_cast<uintptr_t>(f.w[r]) |
         reinterpret_cast<uintptr_t>(f.y[r])) & 1u)
      return false;
    if (f.bias && (reinterpret_cast<uintptr_t>(f.bias[r]) & bias_align)) return false;
  }
  return true;
}

cudaError_t read_fault_word3(int32_t* code, int clear) {
  cudaError_t e = cudaMemcpyFromSymbol(code, g_bra_fault_word3, sizeof(int32_t));
  if (e != cudaSuccess) return e;
  if (clear) {
    const int32_t z = 0;
    e = cudaMemcpyToSymbol(g_bra_fault_word3, &z, sizeof(int32_t));
  }
  return e;
}

}  // namespace bra
