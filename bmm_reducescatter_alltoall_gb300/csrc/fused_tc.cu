// Tensor-core fused BMM -> TP ReduceScatter -> bias Add -> EP AllToAll for
// sm_103a, one CTA per 128 x 256 output tile: TMA loads into 128-byte-swizzled
// shared memory, tcgen05.mma with the fp32 accumulator in tensor memory, and
// an epilogue that writes each element straight to its final all-to-all
// destination.  (fused_tc2.cu is the CTA-pair form with 256 x 256 tiles.)
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
//                      64x64 B boxes (B is the weight, N-contiguous; one
//                      64x256 K-major box when the weight is stored
//                      transposed) into a 4-stage ring guarded by full/empty
//                      mbarriers.
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
#include <cstring>
#include <memory>
#include <mutex>

#include "tcu_epilogue.cuh"

namespace bra {

__device__ int32_t g_bra_fault_word = 0;

namespace {

using namespace tc;

#ifndef BRA_TC_STAGES
#define BRA_TC_STAGES 4
#endif
#ifndef BRA_TC_GROUP_M
#define BRA_TC_GROUP_M 16
#endif
constexpr int BM = 128, BN = 256, BK = 64, STAGES = BRA_TC_STAGES;
constexpr int kGroupM = BRA_TC_GROUP_M;
constexpr int A_BYTES = BM * BK * 2;              // 16 KiB
constexpr int B_BOX_BYTES = 64 * BK * 2;          // one 64(N) x 64(K) box, 8 KiB
constexpr int B_BYTES = BN * BK * 2;              // 32 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;    // 48 KiB
constexpr int THREADS = 256;
constexpr int EPI_WARP0 = 4;
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 4 * kEpiStageBytes + 1024;
static_assert(kUStageBytes <= kEpiStageBytes, "element epilogue staging");

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
  int32_t* fault = &g_bra_fault_word;
  // epilogue staging tiles (one per epilogue warp) after the barrier block
  const uint32_t epi_stage_base = bar_base + BAR_BYTES;

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
    tmem_alloc<1>(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish<1>();
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
      const TileCoord tc = tile_coord(tile, p.m_tiles, p.n_tiles, kGroupM);
      const int sl = tc.g / p.El, e = tc.g % p.El;
      for (int t = 0; ok && t < p.tp; ++t) {
        const int r = sl * p.tp + t;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, fault)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_expect_tx(fb, STAGE_BYTES);
          const uint32_t a_dst = smem_base + stage * STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          tma_load_3d(a_dst, &p.tx[r], fb, kb * BK, tc.mt * BM, e);
          if (p.b_kmajor) {
            tma_load_3d(b_dst, &p.tw[r], fb, kb * BK, tc.nt * BN, e);   // BN rows x 128 B
          } else {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_3d(b_dst + c * B_BOX_BYTES, &p.tw[r], fb, tc.nt * BN + c * 64, kb * BK, e);
          }
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
    const RingDescs rd = ring_descs(p, smem_base, smem_base + A_BYTES);
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
          tc_mma<1>(d_tmem, rd.a0 + so + 2 * k, rd.b0 + so + rd.b_kstep * k, p.idesc,
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
  } else if (warp >= EPI_WARP0) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;                      // TMEM lane quarter
    const uint32_t epi_stage = epi_stage_base + (uint32_t)q * kEpiStageBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      const TileCoord tc = tile_coord(tile, p.m_tiles, p.n_tiles, kGroupM);
      const int sl = tc.g / p.El, e = tc.g % p.El;
      // The whole warp leaves together if any lane's wait gave up, so the
      // warp-wide tcgen05.ld always runs on all 32 lanes.
      const bool waited = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, fault);
      if (!__all_sync(0xffffffffu, waited)) break;
      tc_fence_after();
      const uint32_t t_base = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      if (p.y_elem)   // outputs or bias without 16-byte alignment: element stores
        epilogue_rows_u<T, true>(p, t_base, tc.mt * BM + q * 32, sl, e, tc.nt * BN,
                                 bars + BAR_BYTES + q * kEpiStageBytes, lane);
      else
        epilogue_rows<T, BN>(p, t_base, tc.mt * BM + q * 32, sl, e, tc.nt * BN, epi_stage, lane);
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
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc<1>(tmem_base, TMEM_COLS);
  }
}

struct DeviceInfo {
  int sms = 0;
  bool attr_set = false;
};

}  // namespace

bool fused_tc_eligible(const FusedProblem& f) {
  // TMA needs x and weight rows with a 16-byte pitch and 16-byte pointers
  // (the row lengths themselves may be ragged: coordinates past a row's end
  // read zeros); outputs and bias need only element alignment (the epilogue
  // stores element by element when they are not 16-byte aligned).
  if (f.xp % 8 != 0 || f.wp % 8 != 0) return false;
  const int P = f.ep * f.tp;
  if (P > kMaxRanks) return false;
  auto al = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  const uintptr_t bias_align = f.dtype == BRA_BF16 ? 3u : 1u;
  for (int r = 0; r < P; ++r) {
    if (!al(f.x[r]) || !al(f.w[r])) return false;
    if (reinterpret_cast<uintptr_t>(f.y[r]) & 1u) return false;
    if (f.bias && (reinterpret_cast<uintptr_t>(f.bias[r]) & bias_align)) return false;
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
  fill_common(p.get(), f, BM, BN, BK);
  const bool bf16 = f.dtype == BRA_BF16;
  p->idesc = make_idesc(bf16, BM, BN, f.wt != 0);
  p->b_lbo = B_BOX_BYTES;   // next 64-wide N group
  p->b_sbo = 1024;          // next 8 K rows
  const int s_per_launch = kChunkRanks / f.tp > 0 ? kChunkRanks / f.tp : 1;
  for (int s0 = 0; s0 < f.ep; s0 += s_per_launch) {
    const int s1 = s0 + s_per_launch < f.ep ? s0 + s_per_launch : f.ep;
    if (!fill_chunk(p.get(), f, s0, s1, BM, 64, BK, BN)) return cudaErrorInvalidValue;
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

namespace {
// Diagnostic: one bounded wait (the tensor-core kernels' helper) on a
// barrier nothing arrives at; it runs out, records BRA_ERR_TIMEOUT in this
// file's fault word and returns; *status gets the outcome.
__global__ void tc_wait_probe_kernel(int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool done = mbar_wait(smem_u32(&bar), 0, &abort_flag, &g_bra_fault_word);
    *status = done ? BRA_OK : BRA_ERR_TIMEOUT;
  }
}
}  // namespace

cudaError_t launch_tc_wait_probe(int32_t* status, cudaStream_t st) {
  tc_wait_probe_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
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
