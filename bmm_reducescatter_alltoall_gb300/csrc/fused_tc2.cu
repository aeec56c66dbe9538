// CTA-pair form of the tensor-core fused BMM -> TP ReduceScatter -> bias Add
// -> EP AllToAll kernel (sm_103a): a cluster of two CTAs computes one
// 256 x 256 (or 256 x 512) output tile with tcgen05.mma.cta_group::2
// (M=256, N=256, K=16; two such MMAs per K step share the A slice for the
// 512-wide tile).
//
// Same dataflow as fused_tc.cu (CANN guide "BatchMatMulReduceScatterAllToAll
// 原理、shape 约束与 aclnn 两段式调用", 功能说明与计算流程): the K loop of a
// tile spans the tp shards t = 0..tp-1 (the reduce-scatter sum, fp32, in t
// order) and the epilogue adds the sender's bias and stores to the all-to-all
// destination.  What changes is the split of one tile over two SMs:
//   * CTA rank r of the pair loads A rows [256*mt + 128r, +128) and, for each
//     N=256 sub-tile, B columns [.. + 128r, +128) of every K block into its
//     own shared memory; the
//     pair MMA reads A by M and B by N from both CTAs, so each SM's shared
//     memory carries 32 KiB per K block instead of 48 KiB for a one-CTA
//     128 x 256 tile (operand reads plus TMA writes fit the shared-memory
//     bandwidth).
//   * Both CTAs' TMA loads complete on the leader's (rank 0) full barrier;
//     the leader posts the expected bytes of both halves.
//   * Only the leader issues MMAs; its commits multicast to the empty and
//     accumulator-full barriers of both CTAs.
//   * Each CTA's epilogue drains its own TMEM (its 128 rows) and arrives on
//     the leader's accumulator-empty barrier (remote arrive for the peer):
//     four warps, one per TMEM lane quarter, or for the wide tile eight, two
//     per quarter with half of the columns each.
//   * TMEM: 512 columns allocated by the pair (tcgen05.alloc.cta_group::2 in
//     both CTAs; both get the same column range): two 256-column
//     accumulators, or one 512-column accumulator for the wide tile.
//   * Optionally two pairs per cluster share each weight box (see CL below).
// Every wait is bounded (about 4 s by %globaltimer) and reports through the
// device fault word; both CTAs always reach the closing cluster barrier and
// free their tensor memory.
#include <cstdlib>
#include <cstring>
#include <memory>
#include <mutex>

#include "tcu_epilogue.cuh"

namespace bra {

__device__ int32_t g_bra_fault_word2 = 0;

namespace {

using namespace tc;

// Tile raster: super-rows of 16 pair tiles (m) walked n tile by n tile.  At
// the power cap 16 ran the bench workload 3% faster than 8 or 4 (1450 vs
// 1408 TFLOP/s over 250-call loops, alternated in one process), at a higher
// SM clock for the same power; in short runs the sizes tie.
#ifndef BRA_TC2_GROUP_M
#define BRA_TC2_GROUP_M 16
#endif
constexpr int BM = 256;                           // rows per pair tile
constexpr int BM_CTA = 128;                       // rows per CTA
constexpr int BK = 64;
constexpr int kGroupM = BRA_TC2_GROUP_M;
constexpr int A_BYTES = BM_CTA * BK * 2;          // 16 KiB
constexpr int B_BOX_BYTES = 64 * BK * 2;          // 8 KiB: 64 N-major columns
constexpr int B_SUB_BYTES = 128 * BK * 2;         // 16 KiB: one CTA's half of N = 256
constexpr int EPI_WARP0 = 4;
// Epilogue warps of the 512-wide tile: 8 (two per TMEM lane quarter, each
// draining half of the columns) or 4.
#ifndef BRA_TC2_EPI_WARPS2
#define BRA_TC2_EPI_WARPS2 8
#endif
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;

// A pair tile is 256 rows x (256 * NSUB) columns: NSUB N=256 MMAs per K step
// share each A slice.  NSUB = 1: 6-stage ring of 32 KiB, two TMEM
// accumulators (epilogue overlaps the next tile).  NSUB = 2: 4-stage ring of
// 48 KiB, one 128 x 512 accumulator per CTA (all of TMEM), a quarter less
// operand traffic per FLOP from L2 and through shared memory.
static_assert(kUStageBytes <= kEpiStageBytes, "element epilogue staging");

template <int NSUB>
struct Shape {
  static constexpr int BN = 256 * NSUB;
  static constexpr int B_BYTES = NSUB * B_SUB_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int NACC = NSUB == 1 ? 2 : 1;
  static constexpr int EPI_WARPS = NSUB == 1 ? 4 : BRA_TC2_EPI_WARPS2;
  static constexpr int EPI_SPLIT = EPI_WARPS / 4;             // column parts of a lane quarter
  static constexpr int THREADS = (EPI_WARP0 + EPI_WARPS) * 32;
  // stages: as many as fit beside the epilogue warps' staging tiles
  static constexpr int STAGES = NSUB == 1 ? 6 : (EPI_WARPS == 8 ? 3 : 4);
  static constexpr int SMEM_BYTES =
      STAGES * STAGE_BYTES + BAR_BYTES + EPI_WARPS * kEpiStageBytes + 1024;
  static_assert(EPI_WARPS == 4 || (EPI_WARPS == 8 && NSUB == 2), "epilogue warps");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// CL pairs per cluster.  CL = 2: the two pairs compute m tiles 2i and 2i+1
// of the same n tile and load each weight box once, multicast to the CTA of
// either pair that holds it (half of the weight's L2 reads); a stage is free
// again once both pairs' MMAs have read it.
template <typename T, int NSUB, int CL>
__global__ void __cluster_dims__(2 * CL, 1, 1) __launch_bounds__(Shape<NSUB>::THREADS, 1)
    fused_tc2_kernel(const __grid_constant__ TcParams p) {
  static_assert(CL == 1 || CL == 2, "pairs per cluster");
  using S = Shape<NSUB>;
  constexpr int STAGES = S::STAGES, STAGE_BYTES = S::STAGE_BYTES, BN = S::BN, NACC = S::NACC;
  constexpr int EPI_SPLIT = S::EPI_SPLIT, BN_EPI = BN / EPI_SPLIT;
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
  int32_t* fault = &g_bra_fault_word2;
  // epilogue staging tiles (one per epilogue warp) after the barrier block
  const uint32_t epi_stage_base = bar_base + BAR_BYTES;
  static_assert(8 * (2 * STAGES + 4) + 16 <= BAR_BYTES, "barrier area");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();      // 0 .. 2 CL - 1
  const uint32_t r2 = rank & 1u;             // CTA within its pair
  const uint32_t lead = rank & ~1u;          // its pair's leader
  const int pc = (int)(rank >> 1);           // pair within the cluster
  // super-tiles: CL m tiles (one per pair) of one n tile, handed out per cluster
  const int cl = blockIdx.x / (2 * CL), ncl = gridDim.x / (2 * CL);
  const int m_super = (p.m_tiles + CL - 1) / CL;
  const int num_super = p.num_tiles / (p.m_tiles * p.n_tiles) * m_super * p.n_tiles;
  constexpr int kGroupS = kGroupM / CL > 0 ? kGroupM / CL : 1;
  constexpr uint16_t kAllCtas = (uint16_t)((1u << (2 * CL)) - 1u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);     // leader: its expect_tx; both halves' bytes
      mbar_init(empty_bar(s), CL);   // one multicast commit per pair and use
    }
    for (int a = 0; a < NACC; ++a) {
      mbar_init(tfull_bar(a), 1);    // one multicast commit per tile
      mbar_init(tempty_bar(a), 2 * S::EPI_WARPS);   // leader: the epilogue warps of each CTA
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
    tmem_alloc<2>(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish<2>();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // barriers of both CTAs initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    const uint32_t leader_full0 = map_to_rank(full_bar(0), lead);
    const uint16_t share = (uint16_t)((1u << rank) | (1u << (rank ^ 2u)));   // CL = 2
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int st = cl; ok && st < num_super; st += ncl) {
      TileCoord tc = tile_coord(st, m_super, p.n_tiles, kGroupS);
      tc.mt = tc.mt * CL + pc;
      const int sl = tc.g / p.El, e = tc.g % p.El;
      const int a_row = tc.mt * BM + (int)r2 * BM_CTA;
      for (int t = 0; ok && t < p.tp; ++t) {
        const int r = sl * p.tp + t;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, fault)) {
            ok = false;
            break;
          }
          if (r2 == 0) mbar_expect_tx(full_bar(stage), 2 * STAGE_BYTES);
          const uint32_t fb = leader_full0 + 8u * stage;
          const uint32_t a_dst = smem_base + stage * STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          tma_load_3d_pair(a_dst, &p.tx[r], fb, kb * BK, a_row, e);
#pragma unroll
          for (int sub = 0; sub < NSUB; ++sub) {
            // this CTA's 128 columns of N=256 sub-tile `sub`
            const int b_col = tc.nt * BN + sub * 256 + (int)r2 * 128;
            const uint32_t bs = b_dst + sub * B_SUB_BYTES;
            if (p.b_kmajor) {
              // 128 rows x 128 B; shared: the pair whose index is sub % 2 loads it
              if (CL == 1)
                tma_load_3d_pair(bs, &p.tw[r], fb, kb * BK, b_col, e);
              else if (sub % 2 == pc)
                tma_load_3d_pair_mc(bs, &p.tw[r], fb, kb * BK, b_col, e, share);
            } else {
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                if (CL == 1)
                  tma_load_3d_pair(bs + c * B_BOX_BYTES, &p.tw[r], fb, b_col + c * 64, kb * BK, e);
                else if ((sub * 2 + c) % 2 == pc)   // boxes dealt over the two pairs
                  tma_load_3d_pair_mc(bs + c * B_BOX_BYTES, &p.tw[r], fb, b_col + c * 64,
                                      kb * BK, e, share);
              }
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    if (!ok) spin_ns(2000000ull);   // let copies already issued land
  } else if (warp == 1 && lane == 0 && r2 == 0) {
    // ---------------- MMA issuer (leader only) ----------------
    const RingDescs rd = ring_descs(p, smem_base, smem_base + A_BYTES);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int st = cl; ok && st < num_super; st += ncl) {
      if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, fault)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);   // acc = 0 when NACC = 1
      const int kk_total = p.tp * p.k_blocks;
      for (int kk = 0; kk < kk_total; ++kk) {
        if (!mbar_wait(full_bar(stage), phase, abort_flag, fault)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t so = (uint64_t)((stage * STAGE_BYTES) >> 4);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
#pragma unroll
          for (int sub = 0; sub < NSUB; ++sub)
            tc_mma<2>(d_tmem + sub * 256, rd.a0 + so + 2 * k,
                      rd.b0 + so + (uint64_t)((sub * B_SUB_BYTES) >> 4) + rd.b_kstep * k, p.idesc,
                      (kk > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit_pair(empty_bar(stage), kAllCtas);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit_pair(tfull_bar(acc), (uint16_t)(0x3u << (2 * pc)));
      if (++acc == NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok) spin_ns(2000000ull);   // let MMAs already issued complete
  } else if (warp >= EPI_WARP0) {
    // ---------------- epilogue (both CTAs) ----------------
    // lane quarter q of TMEM (warp % 4), column part h of EPI_SPLIT
    const int q = warp & 3, h = (warp - EPI_WARP0) >> 2;
    const uint32_t epi_stage = epi_stage_base + (uint32_t)(warp - EPI_WARP0) * kEpiStageBytes;
    const uint32_t leader_tempty0 = map_to_rank(tempty_bar(0), lead);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int st = cl; st < num_super; st += ncl) {
      TileCoord tc = tile_coord(st, m_super, p.n_tiles, kGroupS);
      tc.mt = tc.mt * CL + pc;
      const int sl = tc.g / p.El, e = tc.g % p.El;
      const int row0 = tc.mt * BM + (int)r2 * BM_CTA + q * 32;
      const int n0 = tc.nt * BN + h * BN_EPI;
      // the tile's bias, staged while its accumulator is still being computed
      const bool bias_staged =
          !p.y_elem && epilogue_bias<T, BN_EPI>(p, row0, sl, e, n0, epi_stage, lane);
      const bool waited = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, fault);
      if (!__all_sync(0xffffffffu, waited)) break;
      tc_fence_after();
      const uint32_t t_base = tmem_base + (uint32_t)(acc * BN + h * BN_EPI) +
                              ((uint32_t)(q * 32) << 16);
      // hand the accumulator back to the leader's MMA issuer (remote arrive
      // for the peer) once this warp's TMEM reads are done
      auto release = [&] {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (r2 == 0)
            mbar_arrive(tempty_bar(acc));
          else
            mbar_arrive_cluster(leader_tempty0 + 8u * acc);
        }
      };
      if (p.y_elem) {   // outputs or bias without 16-byte alignment: element stores
        uint8_t* stg = bars + BAR_BYTES + (warp - EPI_WARP0) * kEpiStageBytes;
#pragma unroll 1
        for (int sub = 0; sub < BN_EPI / 256; ++sub)
          epilogue_rows_u<T, true>(p, t_base + sub * 256, row0, sl, e, n0 + sub * 256, stg, lane);
        release();
      } else {
        epilogue_body<T, BN_EPI>(p, t_base, row0, sl, e, n0, epi_stage, lane, bias_staged, release);
      }
      if (++acc == NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // no remote arrive or MMA of the pair still pending
  if (threadIdx.x == 0 && p.status && *abort_flag) atomicExch(p.status, (int32_t)BRA_ERR_TIMEOUT);
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc<2>(tmem_base, TMEM_COLS);
  }
}

struct DeviceInfo2 {
  int clusters[2][2] = {};   // co-resident clusters: [N = 512 tiles][two pairs a cluster]
  bool ready = false;
};

template <typename T, int NSUB, int CL>
cudaError_t setup_kernel(int* clusters) {
  constexpr int smem = Shape<NSUB>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(fused_tc2_kernel<T, NSUB, CL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * CL, 1, 1);
  cfg.blockDim = dim3(Shape<NSUB>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2 * CL;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, fused_tc2_kernel<T, NSUB, CL>, &cfg);
  if (e != cudaSuccess) return e;
  *clusters = n;
  return cudaSuccess;
}

}  // namespace

// Pair tile width.  The 512-wide tile moves a quarter less operand traffic
// per FLOP from L2 and into shared memory, which at the power cap buys a
// higher SM clock (1537 against 1290 MHz on the fp16 M = 8192 workload), but
// its single accumulator leaves the tensor core idle while the epilogue
// drains it.  With a long K loop the clock wins: K = tp * Kp = 8192 ran 5%
// faster sustained and 3-5% in short runs; at K = 4096 (the bf16 M = 4096
// workload) the 256-wide tile with its overlapped epilogue stayed 4-7% ahead.
// BRA_TC2_WIDE=0|1, read at every call, forces the 256- or 512-wide tile.
int fused_tc2_tile_n(const FusedProblem& f) {
  const char* v = std::getenv("BRA_TC2_WIDE");
  if (v && *v) return *v == '1' ? 512 : 256;
  const int64_t K = (int64_t)f.tp * f.Kp;
  const int64_t rows = (int64_t)f.ep * f.C;
  const int64_t tiles = (int64_t)f.ep * f.El * ((rows + 255) / 256) * (((int64_t)f.H + 511) / 512);
  return K >= 8192 && f.H >= 1024 && tiles >= 38 ? 512 : 256;
}

// Whether two pairs share each weight box (clusters of four CTAs).
// BRA_TC2_SHARE=0|1, read at every call, forces the choice.
#ifndef BRA_TC2_SHARE_DEFAULT
#define BRA_TC2_SHARE_DEFAULT 0
#endif
int fused_tc2_share(const FusedProblem&) {
  const char* v = std::getenv("BRA_TC2_SHARE");
  if (v && *v) return *v == '1' ? 1 : 0;
  return BRA_TC2_SHARE_DEFAULT;
}

namespace {

template <int NSUB, int CL>
cudaError_t launch_nsub(const FusedProblem& f, int clusters, cudaStream_t st) {
  using S = Shape<NSUB>;
  std::unique_ptr<TcParams> p(new TcParams);
  std::memset(p.get(), 0, sizeof(TcParams));
  fill_common(p.get(), f, BM, S::BN, BK);
  const bool bf16 = f.dtype == BRA_BF16;
  p->idesc = make_idesc(bf16, BM, 256, f.wt != 0);
  p->b_lbo = B_BOX_BYTES;
  p->b_sbo = 1024;
  const int s_per_launch = kChunkRanks / f.tp > 0 ? kChunkRanks / f.tp : 1;
  for (int s0 = 0; s0 < f.ep; s0 += s_per_launch) {
    const int s1 = s0 + s_per_launch < f.ep ? s0 + s_per_launch : f.ep;
    if (!fill_chunk(p.get(), f, s0, s1, BM_CTA, 64, BK, 128)) return cudaErrorInvalidValue;
    p->num_tiles = (s1 - s0) * f.El * p->m_tiles * p->n_tiles;
    const int num_super = (s1 - s0) * f.El * ((p->m_tiles + CL - 1) / CL) * p->n_tiles;
    const int nc = num_super < clusters ? num_super : clusters;
    if (bf16)
      fused_tc2_kernel<__nv_bfloat16, NSUB, CL><<<2 * CL * nc, S::THREADS, S::SMEM_BYTES, st>>>(*p);
    else
      fused_tc2_kernel<__half, NSUB, CL><<<2 * CL * nc, S::THREADS, S::SMEM_BYTES, st>>>(*p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_fused_tc2(const FusedProblem& f, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static DeviceInfo2 info[64];
  int cl[2][2];
  {
    std::lock_guard<std::mutex> lk(mu);
    DeviceInfo2& di = info[dev & 63];
    if (!di.ready) {
      int a[8] = {};
      if ((e = setup_kernel<__half, 1, 1>(&a[0])) != cudaSuccess) return e;
      if ((e = setup_kernel<__nv_bfloat16, 1, 1>(&a[1])) != cudaSuccess) return e;
      if ((e = setup_kernel<__half, 2, 1>(&a[2])) != cudaSuccess) return e;
      if ((e = setup_kernel<__nv_bfloat16, 2, 1>(&a[3])) != cudaSuccess) return e;
      if ((e = setup_kernel<__half, 1, 2>(&a[4])) != cudaSuccess) return e;
      if ((e = setup_kernel<__nv_bfloat16, 1, 2>(&a[5])) != cudaSuccess) return e;
      if ((e = setup_kernel<__half, 2, 2>(&a[6])) != cudaSuccess) return e;
      if ((e = setup_kernel<__nv_bfloat16, 2, 2>(&a[7])) != cudaSuccess) return e;
      // a[2k], a[2k+1]: the fp16 and bf16 kernels of tile width k % 2, k / 2 + 1 pairs
      for (int k = 0; k < 4; ++k) {
        const int m = a[2 * k] < a[2 * k + 1] ? a[2 * k] : a[2 * k + 1];
        di.clusters[k % 2][k / 2] = m < 1 ? 1 : m;
      }
      di.ready = true;
    }
    for (int k = 0; k < 4; ++k) cl[k % 2][k / 2] = di.clusters[k % 2][k / 2];
  }
  const bool wide = fused_tc2_tile_n(f) == 512;
  if (fused_tc2_share(f))
    return wide ? launch_nsub<2, 2>(f, cl[1][1], st) : launch_nsub<1, 2>(f, cl[0][1], st);
  return wide ? launch_nsub<2, 1>(f, cl[1][0], st) : launch_nsub<1, 1>(f, cl[0][0], st);
}

cudaError_t read_fault_word2(int32_t* code, int clear) {
  cudaError_t e = cudaMemcpyFromSymbol(code, g_bra_fault_word2, sizeof(int32_t));
  if (e != cudaSuccess) return e;
  if (clear) {
    const int32_t z = 0;
    e = cudaMemcpyToSymbol(g_bra_fault_word2, &z, sizeof(int32_t));
  }
  return e;
}

}  // namespace bra
