// Tensor-core fused BMM -> TP ReduceScatter -> bias Add -> EP AllToAll for
// rows that are not 16-byte aligned (M/tp, H or H/tp not a multiple of 8
// elements, or element-aligned pointers), fed by TMA (sm_103a, CTA pair).
//
// Dataflow as in fused_tc2.cu (CANN guide "BatchMatMulReduceScatterAllToAll
// 原理、shape 约束与 aclnn 两段式调用", 功能说明与计算流程): a cluster of two
// CTAs computes a 256 x 256 output tile of Z_{s,e} with
// tcgen05.mma.cta_group::2; the K loop runs over the tp shards (the
// reduce-scatter sum, fp32, in t order) and 64-wide K blocks; the epilogue
// adds the sender's bias, rounds once and stores each element at its
// all-to-all destination (tcu_epilogue.cuh: rows of any alignment).
//
// TMA needs row pitches that are multiples of 16 bytes.  A row-major matrix
// whose pitch is not is split into row classes: with n = the least power of
// two for which n rows span a multiple of 16 bytes, rows q, q+n, q+2n, ...
// form class q, a 2-D tensor with a legal pitch (n rows) whose rows all
// start at the same offset (delta_q elements) past a 16-byte boundary.  One
// map per class starts at the boundary below its first row, so a box loaded
// at an aligned inner coordinate x holds the row's elements from x - delta_q
// on; the boxes are 8 elements wider than the tile so that every element of
// the tile is inside.  Per CTA and K block that is n_x boxes of A rows and
// n_w boxes of B rows (B rows are K rows of a (Kp, H) weight, or N rows of a
// transposed (H, Kp) weight) into a raw stage, without swizzle.
//
// Roles (one CTA; both CTAs of the pair run all of them):
//   warp 0 (one lane)   TMA producer: raw A and B boxes of each K block into a
//                       RAW_STAGES-deep ring (raw_full / raw_empty).
//   warp 1              allocates 512 TMEM columns (two 256-column fp32
//                       accumulators per CTA); in the leader its lane 0
//                       issues the pair MMAs (M=256, N=256, K=16) and
//                       commits to both CTAs.
//   warps 2..           realign (RGROUPS groups of RWARPS warps, taking K
//                       blocks in turn): shift each raw row into the
//                       128-byte-swizzle layout a TMA box would have produced,
//                       by the class's delta (a compile-time shift picked per
//                       batch: the rows a warp moves at once share a class),
//                       and zero the weight's K rows past Kp.  A warp frees
//                       the raw stage once its rows are in registers, waits
//                       for the canonical slot (SW_STAGES-deep ring), stores,
//                       and runs fence.proxy.async; the group then meets at a
//                       named barrier and publishes the stage: the leader's
//                       group on its own sw_full, the peer's group on a local
//                       `ready` barrier.  Eight lanes move one row's 128
//                       bytes, so reads and writes are free of bank conflicts.
//   warps SIG_WARP0..   in the peer CTA, signal warps take stages in turn: on
//                       `ready`, one release arrive at cluster scope on the
//                       leader's sw_full (such an arrive takes ~2k cycles, so
//                       several are kept in flight, off the realign path).
//   warps EPI_WARP0..+3 epilogue of the CTA's 128 accumulator rows.
// Every wait is bounded (about 4 s); a wait that runs out records
// BRA_ERR_TIMEOUT in a device word and every role leaves its loop; both CTAs
// reach the closing cluster barrier and free their tensor memory.
#include <cstring>
#include <memory>
#include <mutex>

#include "tcu_epilogue.cuh"

namespace bra {

__device__ int32_t g_bra_fault_word4 = 0;

namespace {

using namespace tc;

#ifndef BRA_TCR_RWARPS
#define BRA_TCR_RWARPS 8
#endif
#ifndef BRA_TCR_RGROUPS
#define BRA_TCR_RGROUPS 1
#endif
#ifndef BRA_TCR_RAW_STAGES
#define BRA_TCR_RAW_STAGES 3
#endif
#ifndef BRA_TCR_SW_STAGES
#define BRA_TCR_SW_STAGES 3
#endif
constexpr int BM = 256, BM_CTA = 128, BN = 256, BN_CTA = 128, BK = 64;
constexpr int kGroupM = 8;
constexpr int RWARPS = BRA_TCR_RWARPS;       // realign warps per group
constexpr int RGROUPS = BRA_TCR_RGROUPS;     // groups take K blocks in turn
constexpr int RAW_STAGES = BRA_TCR_RAW_STAGES, SW_STAGES = BRA_TCR_SW_STAGES;
constexpr int TMA_WARP = 0, MMA_WARP = 1, RW0 = 2;
// Warps between the realign warps and the epilogue signal the leader for the
// peer CTA (at least two, taking stages in turn).
constexpr int SIG_WARP0 = RW0 + RGROUPS * RWARPS;
constexpr int EPI_WARP0 = ((SIG_WARP0 + 2 + 3) / 4) * 4;   // lane quarter = warp % 4
constexpr int NSIG = EPI_WARP0 - SIG_WARP0;
constexpr int NBW = 16 / RWARPS;                           // realign batches per warp and stage
static_assert(16 % RWARPS == 0, "realign batches");
constexpr int THREADS = (EPI_WARP0 + 4) * 32;
// canonical stage: A 128 x 64 K-major; B 64 x 128 N-major (two 64 x 64 boxes)
// or, transposed weight, 128 x 64 K-major
constexpr int A_BYTES = BM_CTA * BK * 2;          // 16 KiB
constexpr int B_BOX_BYTES = 64 * BK * 2;          // 8 KiB
constexpr int B_BYTES = BN_CTA * BK * 2;          // 16 KiB
constexpr int SW_BYTES = A_BYTES + B_BYTES;       // 32 KiB
// raw stage: rows 8 elements wider than the tile
constexpr int KROW = (BK + 8) * 2;                // 144 bytes: 72 K elements
constexpr int NROW = (BN_CTA + 8) * 2;            // 272 bytes: 136 N elements
constexpr int RAW_A = BM_CTA * KROW;              // 18 KiB
constexpr int RAW_B = BN_CTA * KROW;              // 18 KiB, >= BK * NROW
constexpr int RAW_BYTES = RAW_A + RAW_B;
static_assert(BK * NROW <= RAW_B, "raw B");
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES =
    SW_STAGES * SW_BYTES + RAW_STAGES * RAW_BYTES + BAR_BYTES + 4 * kUStageBytes + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
// Class maps per launch: each rank of the launch has n_x + n_w of them.
constexpr int kRMaps = 176;

struct RParams {
  CUtensorMap maps[kRMaps];    // rank-local index rl: x classes at rl*(ncx+ncw), then w classes
  const void* bias[kChunkRanks];
  void* y[kMaxRanks];
  int8_t delta[kRMaps];        // class map's row offset in elements; -1: the class has no row
  int ep, tp, El, C, Kp, H, type, has_bias;
  int s0;                      // first source EP rank of this launch
  int nranks;
  int rows;                    // ep * C
  int m_tiles, n_tiles, k_blocks, num_tiles;
  int b_kmajor;                // weight stored transposed: B rows are N rows
  int lgx, lgw;                // log2 of the class counts of x rows and weight rows
  uint32_t idesc;
  int32_t* status;             // per-call timeout word (optional)
};
static_assert(sizeof(RParams) <= 32764, "kernel parameter space");

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Wait on a barrier that CTAs of the cluster arrive on (acquire at cluster
// scope); bounded as mbar_wait.
__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __noinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, int32_t* fault_word) {
  if (mbar_try_cluster(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int k = 0; k < 64; ++k)
      if (mbar_try_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitTimeoutNs) {
      *abort_flag = 1;
      atomicExch(fault_word, (int32_t)BRA_ERR_TIMEOUT);
      return false;
    }
  }
}

// One realign batch: four warp steps of one class box, each lane moving one
// 16-byte chunk per step: o[s] = the 16 bytes that start D elements (2D
// bytes) into the raw granule pair at src[s], or zeros where bit s of `zero`
// is set.  All loads are issued before the first is used.
template <int D>
__device__ __forceinline__ void shift_batch(const uint32_t (&src)[4], uint32_t zero,
                                            uint4 (&o)[4]) {
  uint4 a[4], b[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    a[s] = lds128e(src[s]);
    if constexpr (D != 0) b[s] = lds128e(src[s] + 16);
  }
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    if constexpr (D == 0) {
      o[s] = a[s];
    } else {
      const uint32_t x[8] = {a[s].x, a[s].y, a[s].z, a[s].w, b[s].x, b[s].y, b[s].z, b[s].w};
      constexpr int w = D / 2;
      if constexpr (D % 2 == 0) {
        o[s] = make_uint4(x[w], x[w + 1], x[w + 2], x[w + 3]);
      } else {
        o[s].x = __funnelshift_r(x[w], x[w + 1], 16);
        o[s].y = __funnelshift_r(x[w + 1], x[w + 2], 16);
        o[s].z = __funnelshift_r(x[w + 2], x[w + 3], 16);
        o[s].w = __funnelshift_r(x[w + 3], x[w + 4], 16);
      }
    }
    if ((zero >> s) & 1u) o[s] = make_uint4(0u, 0u, 0u, 0u);
  }
}
__device__ __forceinline__ void shift_batch_rt(int d, const uint32_t (&src)[4], uint32_t zero,
                                               uint4 (&o)[4]) {
  switch (d) {
    case 1: shift_batch<1>(src, zero, o); break;
    case 2: shift_batch<2>(src, zero, o); break;
    case 3: shift_batch<3>(src, zero, o); break;
    case 4: shift_batch<4>(src, zero, o); break;
    case 5: shift_batch<5>(src, zero, o); break;
    case 6: shift_batch<6>(src, zero, o); break;
    case 7: shift_batch<7>(src, zero, o); break;
    default: shift_batch<0>(src, zero, o); break;
  }
}

// Named barrier of realign group g (id 1 + g) as a reduction: true on every
// thread of the group iff v is true on all of them.  Every thread of the
// group reaches each use, since the group leaves its loop only as a whole.
__device__ __forceinline__ bool realign_all(int g, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(1 + g), "n"(RWARPS * 32)
      : "memory");
  return r != 0;
}

template <typename T>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    fused_tcr_kernel(const __grid_constant__ RParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sw_base = smem_u32(smem);
  const uint32_t raw_base = sw_base + SW_STAGES * SW_BYTES;
  uint8_t* bars = smem + SW_STAGES * SW_BYTES + RAW_STAGES * RAW_BYTES;
  const uint32_t bar_base = smem_u32(bars);
  constexpr int NB = 2 * RAW_STAGES + 3 * SW_STAGES;
  auto raw_full = [&](int s) { return bar_base + 8u * s; };
  auto raw_empty = [&](int s) { return bar_base + 8u * (RAW_STAGES + s); };
  auto sw_full = [&](int s) { return bar_base + 8u * (2 * RAW_STAGES + s); };
  auto sw_empty = [&](int s) { return bar_base + 8u * (2 * RAW_STAGES + SW_STAGES + s); };
  auto ready = [&](int s) { return bar_base + 8u * (2 * RAW_STAGES + 2 * SW_STAGES + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (NB + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (NB + 2 + a); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8 * (NB + 4));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 8 * (NB + 4) + 8);
  static_assert(8 * (NB + 4) + 16 <= BAR_BYTES, "barrier area");
  int32_t* fault = &g_bra_fault_word4;
  uint8_t* epi_smem = bars + BAR_BYTES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int ncx = 1 << p.lgx, ncw = 1 << p.lgw, mpr = ncx + ncw;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RAW_STAGES; ++s) {
      mbar_init(raw_full(s), 1);            // expect_tx of this CTA's producer
      mbar_init(raw_empty(s), RWARPS);      // each realign warp of the stage's group
    }
    for (int s = 0; s < SW_STAGES; ++s) {
      mbar_init(sw_full(s), 2);             // leader: one arrival per CTA of the pair
      mbar_init(sw_empty(s), 1);            // one multicast commit per use
      mbar_init(ready(s), 1);               // peer: its realign group is done
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 8);          // leader: 4 epilogue warps of each CTA
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == TMA_WARP && lane == 0)
    for (int i = 0; i < p.nranks * mpr; ++i)
      if (p.delta[i] >= 0) tma_prefetch_desc(&p.maps[i]);   // classes with rows only
  if (warp == MMA_WARP) {
    tmem_alloc<2>(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish<2>();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // barriers of both CTAs initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == TMA_WARP) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < p.num_tiles; tile += npairs) {
        const TileCoord tc = tile_coord(tile, p.m_tiles, p.n_tiles, kGroupM);
        const int sl = tc.g / p.El, e = tc.g % p.El;
        // first flat row (over all local experts) of this CTA's A rows and,
        // for a transposed weight, of its B rows
        const int fa = e * p.rows + tc.mt * BM + (int)rank * BM_CTA;
        const int fbn = e * p.H + tc.nt * BN + (int)rank * BN_CTA;
        const int bcol = tc.nt * BN + (int)rank * BN_CTA;
        for (int t = 0; ok && t < p.tp; ++t) {
          const int rl = sl * p.tp + t;
          const CUtensorMap* xm = &p.maps[rl * mpr];
          const CUtensorMap* wm = xm + ncx;
          const int8_t* xd = &p.delta[rl * mpr];
          const int8_t* wd = xd + ncx;
          uint32_t bytes = 0;
          for (int q = 0; q < ncx; ++q)
            if (xd[q] >= 0) bytes += (uint32_t)(RAW_A >> p.lgx);
          for (int q = 0; q < ncw; ++q)
            if (wd[q] >= 0) bytes += (uint32_t)((p.b_kmajor ? RAW_B : BK * NROW) >> p.lgw);
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!mbar_wait(raw_empty(stage), phase ^ 1u, abort_flag, fault)) {
              ok = false;
              break;
            }
            const uint32_t fb = raw_full(stage);
            mbar_expect_tx(fb, bytes);
            const uint32_t ra = raw_base + stage * RAW_BYTES, rb = ra + RAW_A;
            const int k0 = kb * BK;
            for (int b = 0; b < ncx; ++b) {
              const int R = fa + b, q = R & (ncx - 1);
              if (xd[q] >= 0) tma_load_2d(ra + b * (RAW_A >> p.lgx), &xm[q], fb, k0, R >> p.lgx);
            }
            if (p.b_kmajor) {
              for (int b = 0; b < ncw; ++b) {
                const int R = fbn + b, q = R & (ncw - 1);
                if (wd[q] >= 0) tma_load_2d(rb + b * (RAW_B >> p.lgw), &wm[q], fb, k0, R >> p.lgw);
              }
            } else {
              const int fbk = e * p.Kp + k0;
              for (int b = 0; b < ncw; ++b) {
                const int R = fbk + b, q = R & (ncw - 1);
                if (wd[q] >= 0)
                  tma_load_2d(rb + b * ((BK * NROW) >> p.lgw), &wm[q], fb, bcol, R >> p.lgw);
              }
            }
            if (++stage == RAW_STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) spin_ns(2000000ull);   // let copies already issued land
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (leader only) ----------------
      const uint64_t a0 = smem_desc_sw128(sw_base, 16, 1024);
      const uint64_t b0 = p.b_kmajor ? smem_desc_sw128(sw_base + A_BYTES, 16, 1024)
                                     : smem_desc_sw128(sw_base + A_BYTES, B_BOX_BYTES, 1024);
      const uint32_t b_kstep = p.b_kmajor ? 2u : 128u;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < p.num_tiles; tile += npairs) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, fault)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        const int kk_total = p.tp * p.k_blocks;
        for (int kk = 0; kk < kk_total; ++kk) {
          if (!mbar_wait_cluster(sw_full(stage), phase, abort_flag, fault)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t so = (uint64_t)((stage * SW_BYTES) >> 4);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma<2>(d_tmem, a0 + so + 2 * k, b0 + so + b_kstep * k, p.idesc,
                      (kk > 0 || k > 0) ? 1u : 0u);
          tc_commit_pair(sw_empty(stage), 0x3);
          if (++stage == SW_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair(tfull_bar(acc), 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) spin_ns(2000000ull);   // let MMAs already issued complete
    }
  } else if (warp >= RW0 && warp < RW0 + RGROUPS * RWARPS) {
    // ---------------- realign (both CTAs) ----------------
    // 64 warp steps per K block (32 for A, 32 for B) in 16 batches of four
    // steps inside one class box; group g takes the K blocks n with
    // n % RGROUPS == g (n counts the CTA's K blocks), and its warp rw the
    // batches rw, rw + RWARPS, ...  A warp frees the raw stage as soon as its
    // rows are in registers, then waits for the canonical slot.
    const int grp = (warp - RW0) / RWARPS, rw = (warp - RW0) % RWARPS;
    int n = 0;
    const int rg = lane >> 3, c = lane & 7;
    const int sx = 5 - p.lgx, sw = 5 - p.lgw;   // log2 of warp steps per class box
    int rs = 0, ss = 0;
    uint32_t rph = 0, sph = 0;
    bool ok = true;
    for (int tile = pair; ok && tile < p.num_tiles; tile += npairs) {
      const TileCoord tc = tile_coord(tile, p.m_tiles, p.n_tiles, kGroupM);
      const int sl = tc.g / p.El, e = tc.g % p.El;
      const int fa = e * p.rows + tc.mt * BM + (int)rank * BM_CTA;
      const int fbn = e * p.H + tc.nt * BN + (int)rank * BN_CTA;
      for (int t = 0; ok && t < p.tp; ++t) {
        const int rl = sl * p.tp + t;
        const int8_t* xd = &p.delta[rl * mpr];
        const int8_t* wd = xd + ncx;
        for (int kb = 0; kb < p.k_blocks; ++kb, ++n) {
          if (n % RGROUPS == grp) {
            // all warps of the group go on, or all leave (a wait that gave up)
            if (!realign_all(grp, mbar_wait(raw_full(rs), rph, abort_flag, fault))) {
              ok = false;
              break;
            }
            const uint32_t ra = raw_base + rs * RAW_BYTES, rb = ra + RAW_A;
            const uint32_t sa = sw_base + ss * SW_BYTES, sb = sa + A_BYTES;
            const int k0 = kb * BK;
            const int fbk = e * p.Kp + k0;
            uint4 val[NBW][4];
            uint32_t dst[NBW][4];
#pragma unroll
            for (int h = 0; h < NBW; ++h) {
              const int bt = rw + h * RWARPS;
              uint32_t src[4], zero = 0;
              int d;
              if (bt < 8) {
                // A: rows i = b + n_x * j, eight lanes a row, four rows a step
                const int it0 = bt * 4, b = it0 >> sx, v0 = it0 & ((1 << sx) - 1);
                const uint32_t box = ra + b * (RAW_A >> p.lgx);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                  const int j = 4 * (v0 + s) + rg, i = b + (j << p.lgx);
                  src[s] = box + j * KROW + c * 16;
                  dst[h][s] = sa + i * 128 + ((c ^ (i & 7)) << 4);
                }
                d = xd[(fa + b) & (ncx - 1)];
              } else if (p.b_kmajor) {
                // B, transposed weight: N rows, as A
                const int it0 = (bt - 8) * 4, b = it0 >> sw, v0 = it0 & ((1 << sw) - 1);
                const uint32_t box = rb + b * (RAW_B >> p.lgw);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                  const int j = 4 * (v0 + s) + rg, i = b + (j << p.lgw);
                  src[s] = box + j * KROW + c * 16;
                  dst[h][s] = sb + i * 128 + ((c ^ (i & 7)) << 4);
                }
                d = wd[(fbn + b) & (ncw - 1)];
              } else {
                // B, weight (Kp, H): two K rows a step, both 64-column halves;
                // K rows past Kp become zeros
                const int it0 = (bt - 8) * 4, b = it0 >> sw, v0 = it0 & ((1 << sw) - 1);
                const uint32_t box = rb + b * ((BK * NROW) >> p.lgw);
                const int half = rg & 1;
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                  const int j = 2 * (v0 + s) + (rg >> 1), kr = b + (j << p.lgw);
                  src[s] = box + j * NROW + (half * 8 + c) * 16;
                  dst[h][s] = sb + half * B_BOX_BYTES + kr * 128 + ((c ^ (kr & 7)) << 4);
                  if (k0 + kr >= p.Kp) zero |= 1u << s;
                }
                d = wd[(fbk + b) & (ncw - 1)];
              }
              shift_batch_rt(d, src, zero, val[h]);
            }
            // this warp's reads of the raw stage are done
            __syncwarp();
            if (lane == 0) mbar_arrive(raw_empty(rs));
            const bool got = mbar_wait(sw_empty(ss), sph ^ 1u, abort_flag, fault);
            if (got) {
#pragma unroll
              for (int h = 0; h < NBW; ++h)
#pragma unroll
                for (int s = 0; s < 4; ++s) sts128(dst[h][s], val[h][s]);
            }
            // generic-proxy writes -> visible to the tensor core; the barrier
            // also tells the group whether every wait succeeded
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (!realign_all(grp, got)) {
              ok = false;
              break;
            }
            // publish: the leader arrives on its own barrier; the peer tells
            // a signal warp, which makes the release at cluster scope
            if (rw == 0 && lane == 0) mbar_arrive(rank == 0 ? sw_full(ss) : ready(ss));
          }
          if (++rs == RAW_STAGES) {
            rs = 0;
            rph ^= 1u;
          }
          if (++ss == SW_STAGES) {
            ss = 0;
            sph ^= 1u;
          }
        }
      }
    }
  } else if (warp >= SIG_WARP0 && warp < EPI_WARP0) {
    // ---------------- peer signal warps ----------------
    // Signal warp k takes the stages n with n % NSIG == k: once the peer's
    // realign group is done (ready), one release arrive at cluster scope on
    // the leader's sw_full makes those writes visible to the leader's MMA.
    // These arrives take a while each; several warps keep them overlapped.
    if (rank == 1 && lane == 0) {
      const int k = warp - SIG_WARP0;
      const uint32_t leader_sw_full0 = map_to_rank(sw_full(0), 0);
      int n = 0, ss = 0;
      uint32_t sph = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < p.num_tiles; tile += npairs) {
        for (int kk = 0; kk < p.tp * p.k_blocks; ++kk, ++n) {
          if (n % NSIG == k) {
            if (!mbar_wait(ready(ss), sph, abort_flag, fault)) {
              ok = false;
              break;
            }
            mbar_arrive_cluster(leader_sw_full0 + 8u * ss);
          }
          if (++ss == SW_STAGES) {
            ss = 0;
            sph ^= 1u;
          }
        }
      }
    }
  } else if (warp >= EPI_WARP0) {
    // ---------------- epilogue (both CTAs) ----------------
    const int q = warp & 3;
    uint8_t* stg = epi_smem + q * kUStageBytes;
    const uint32_t leader_tempty0 = map_to_rank(tempty_bar(0), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = pair; tile < p.num_tiles; tile += npairs) {
      const TileCoord tc = tile_coord(tile, p.m_tiles, p.n_tiles, kGroupM);
      const int sl = tc.g / p.El, e = tc.g % p.El;
      const bool waited = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, fault);
      if (!__all_sync(0xffffffffu, waited)) break;
      tc_fence_after();
      const uint32_t t_base = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      const int row0 = tc.mt * BM + (int)rank * BM_CTA + q * 32;
      epilogue_rows_u<T, false>(p, t_base, row0, sl, e, tc.nt * BN, stg, lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(tempty_bar(acc));
        else
          mbar_arrive_cluster(leader_tempty0 + 8u * acc);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // no remote arrive or MMA of the pair still pending
  if (threadIdx.x == 0 && p.status && *abort_flag) atomicExch(p.status, (int32_t)BRA_ERR_TIMEOUT);
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc<2>(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
int ilog2(int n) {
  int l = 0;
  while ((1 << l) < n) ++l;
  return l;
}

// Largest delta (elements past a 16-byte boundary) of the first rows of n
// classes, over all base pointers.
int max_delta(int64_t pitch, int n, const void* const* bases, int count) {
  int dmax = 0;
  for (int i = 0; i < count; ++i)
    for (int q = 0; q < n; ++q) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(bases[i]) + (uintptr_t)(q * pitch * 2);
      const int d = (int)((a & 15u) >> 1);
      dmax = d > dmax ? d : dmax;
    }
  return dmax;
}

// Row classes of a row-major 16-bit matrix with rows of `rowlen` elements
// `pitch` elements apart (the row length, or a caller's larger pitch): the
// least power of two n for which n rows span a multiple of 16 bytes and the
// class map's rows (rowlen + delta elements, starting delta before the
// row) do not overlap, n * pitch >= rowlen + delta for every class.  At most
// 8, since 8 * pitch >= rowlen + 7.
int row_classes(int64_t rowlen, int64_t pitch, const void* const* bases, int count) {
  int n = 1;
  while ((pitch * 2 * n) % 16 != 0) n *= 2;
  while (n < 8 && n * pitch < rowlen + max_delta(pitch, n, bases, count)) n *= 2;
  return n;
}

// Class q of the nrows x rowlen matrix at `base`, rows `pitch` elements
// apart (rows q, q+n, ...): a 2-D map starting at the 16-byte boundary at or
// below row q; *delta = the row's offset from it in elements, or -1 when the
// class has no row.  The boundary lies in the same allocation as the matrix
// (allocations start 16-byte aligned), and the map ends at the last row's
// end, so elements between a row's end and the next row are never read.
bool encode_class(CUtensorMap* m, int8_t* delta, const void* base, int64_t rowlen, int64_t pitch,
                  int64_t nrows, int n, int q, uint32_t box0, uint32_t box1) {
  std::memset(m, 0, sizeof(*m));
  if (q >= nrows) {
    *delta = -1;
    return true;
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const uintptr_t a = reinterpret_cast<uintptr_t>(base) + (uintptr_t)(q * pitch * 2);
  const uintptr_t a16 = a & ~(uintptr_t)15;
  const int d = (int)((a - a16) / 2);
  const cuuint64_t dims[2] = {(cuuint64_t)(rowlen + d), (cuuint64_t)((nrows - q + n - 1) / n)};
  const cuuint64_t strides[1] = {(cuuint64_t)(pitch * 2 * n)};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  *delta = (int8_t)d;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, reinterpret_cast<void*>(a16), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Classes {
  int ncx, ncw;
};
Classes classes_of(const FusedProblem& f) {
  const int P = f.ep * f.tp;
  Classes c;
  c.ncx = row_classes(f.Kp, f.xp, f.x, P);
  c.ncw = row_classes(f.wt ? f.Kp : f.H, f.wp, f.w, P);
  return c;
}

struct TcrInfo {
  int pairs = 0;
  bool ready = false;
};

template <typename T>
cudaError_t setup_tcr(int* pairs) {
  cudaError_t e = cudaFuncSetAttribute(fused_tcr_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, fused_tcr_kernel<T>, &cfg);
  if (e != cudaSuccess) return e;
  *pairs = n;
  return cudaSuccess;
}

}  // namespace

bool fused_tcr_eligible(const FusedProblem& f) {
  const int P = f.ep * f.tp;
  if (P > kMaxRanks) return false;
  const uintptr_t bias_align = f.dtype == BRA_BF16 ? 3u : 1u;
  for (int r = 0; r < P; ++r) {
    if ((reinterpret_cast<uintptr_t>(f.x[r]) | reinterpret_cast<uintptr_t>(f.w[r]) |
         reinterpret_cast<uintptr_t>(f.y[r])) & 1u)
      return false;
    if (f.bias && (reinterpret_cast<uintptr_t>(f.bias[r]) & bias_align)) return false;
  }
  // flat row indices and TMA coordinates in int32
  const int64_t x_rows = (int64_t)f.El * f.ep * f.C;
  const int64_t w_rows = (int64_t)f.El * (f.wt ? f.H : f.Kp);
  if (x_rows + BM >= INT32_MAX || w_rows + BN >= INT32_MAX) return false;
  const Classes c = classes_of(f);
  return (c.ncx + c.ncw) * f.tp <= kRMaps;
}

cudaError_t launch_fused_tcr(const FusedProblem& f, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static TcrInfo info[64];
  int pairs = 1;
  {
    std::lock_guard<std::mutex> lk(mu);
    TcrInfo& di = info[dev & 63];
    if (!di.ready) {
      int a = 0, b = 0;
      if ((e = setup_tcr<__half>(&a)) != cudaSuccess) return e;
      if ((e = setup_tcr<__nv_bfloat16>(&b)) != cudaSuccess) return e;
      di.pairs = a < b ? a : b;
      if (di.pairs < 1) di.pairs = 1;
      di.ready = true;
    }
    pairs = di.pairs;
  }
  const Classes cl = classes_of(f);
  const int mpr = cl.ncx + cl.ncw;
  std::unique_ptr<RParams> p(new RParams);
  std::memset(p.get(), 0, sizeof(RParams));
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
  p->lgx = ilog2(cl.ncx);
  p->lgw = ilog2(cl.ncw);
  p->idesc = make_idesc(f.dtype == BRA_BF16, BM, BN, f.wt != 0);
  int ranks_per_launch = kRMaps / mpr;
  if (ranks_per_launch > kChunkRanks) ranks_per_launch = kChunkRanks;
  const int s_per_launch = ranks_per_launch / f.tp;
  if (s_per_launch < 1) return cudaErrorInvalidValue;
  const int64_t x_rows = (int64_t)f.El * f.ep * f.C;
  const int64_t w_rows = (int64_t)f.El * (f.wt ? f.H : f.Kp);
  const int64_t w_len = f.wt ? f.Kp : f.H;
  const uint32_t wbox0 = f.wt ? (uint32_t)(BK + 8) : (uint32_t)(BN_CTA + 8);
  const uint32_t wbox1 = f.wt ? (uint32_t)(BN_CTA / cl.ncw) : (uint32_t)(BK / cl.ncw);
  for (int s0 = 0; s0 < f.ep; s0 += s_per_launch) {
    const int s1 = s0 + s_per_launch < f.ep ? s0 + s_per_launch : f.ep;
    p->s0 = s0;
    p->nranks = (s1 - s0) * f.tp;
    for (int rl = 0; rl < p->nranks; ++rl) {
      const int gr = s0 * f.tp + rl;
      p->bias[rl] = f.bias ? f.bias[gr] : nullptr;
      CUtensorMap* xm = &p->maps[rl * mpr];
      int8_t* xd = &p->delta[rl * mpr];
      for (int q = 0; q < cl.ncx; ++q)
        if (!encode_class(&xm[q], &xd[q], f.x[gr], f.Kp, f.xp, x_rows, cl.ncx, q, BK + 8,
                          BM_CTA / cl.ncx))
          return cudaErrorInvalidValue;
      for (int q = 0; q < cl.ncw; ++q)
        if (!encode_class(&xm[cl.ncx + q], &xd[cl.ncx + q], f.w[gr], w_len, f.wp, w_rows,
                          cl.ncw, q, wbox0, wbox1))
          return cudaErrorInvalidValue;
    }
    p->num_tiles = (s1 - s0) * f.El * p->m_tiles * p->n_tiles;
    const int np = p->num_tiles < pairs ? p->num_tiles : pairs;
    if (f.dtype == BRA_BF16)
      fused_tcr_kernel<__nv_bfloat16><<<2 * np, THREADS, SMEM_BYTES, st>>>(*p);
    else
      fused_tcr_kernel<__half><<<2 * np, THREADS, SMEM_BYTES, st>>>(*p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

namespace {
// Diagnostic: one bounded cluster-scope wait (the helper of this kernel's MMA
// issuer, which waits for both CTAs' stages) on a barrier nothing arrives
// at; it runs out, records BRA_ERR_TIMEOUT in this file's fault word and
// returns; *status gets the outcome.
__global__ void tcr_wait_probe_kernel(int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool done = mbar_wait_cluster(smem_u32(&bar), 0, &abort_flag, &g_bra_fault_word4);
    *status = done ? BRA_OK : BRA_ERR_TIMEOUT;
  }
}
}  // namespace

cudaError_t launch_tcr_wait_probe(int32_t* status, cudaStream_t st) {
  tcr_wait_probe_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

cudaError_t read_fault_word4(int32_t* code, int clear) {
  cudaError_t e = cudaMemcpyFromSymbol(code, g_bra_fault_word4, sizeof(int32_t));
  if (e != cudaSuccess) return e;
  if (clear) {
    const int32_t z = 0;
    e = cudaMemcpyToSymbol(g_bra_fault_word4, &z, sizeof(int32_t));
  }
  return e;
}

}  // namespace bra
