// Indexed all_to_all_v: the URMA indexed exchange of the PyPTO page
// "LowerL2TensorCollectives Pass", §A5 URMA 索引交换.  The page names the
// operands (input, send_counts, recv_counts, index) and says the cores share
// the local data movement before the remote transfers; it leaves `index`
// undefined.  Reading implemented here: rank i's send list is its input
// gathered through its index,
//     send_i[k] = input_i[index_i[k]],   k < n_i = sum_j send_counts[i][j],
// and the send lists are exchanged as in all_to_all_v (same bookkeeping):
//     out_j[recv_displs[j][i] + m] = send_i[send_displs[i][j] + m].
// On one GPU the local movement and the exchange are one pass: each position
// k of a send list is gathered and stored straight at its destination.
//
// Launch width: the page makes core_num L the exact number of cores a launch
// uses.  Here that is L blocks, one per SM (a block of 1024 threads at more
// than 32 registers each holds over half an SM's register file, so no two
// share an SM), at most the SM count.  The block keeps its shared memory
// small: random gathers need the L1 for the lines they have in flight.  The
// blocks split the send lists of ranks 0..P-1, taken one after another, into
// equal position ranges; a block walks its range rank by rank and, inside a rank, by
// destination.  Every block reads the whole count matrix first and rejects
// the call (nothing written) on a negative count or a NULL buffer that would
// be touched, so all blocks take the same decision without talking to each
// other.  In the copy, consecutive threads take consecutive positions: index
// loads and stores are coalesced, the gathers follow the index; each thread
// keeps eight positions in flight (4% faster than four, at 64 registers, no
// spills; 512 threads with eight were 10-17% slower).  An index outside [0, in_len_i) is never
// dereferenced; its position is not delivered and the optional status word
// gets BRA_ERR_INVALID.  There are no waits.
#include <mutex>

#include "bra_internal.h"

namespace bra {

namespace {

constexpr unsigned kFull = 0xffffffffu;
#ifndef BRA_IA2AV_THREADS
#define BRA_IA2AV_THREADS 1024
#endif
constexpr int kThreads = BRA_IA2AV_THREADS;
constexpr int kWarps = kThreads / 32;
#ifndef BRA_IA2AV_UNROLL
#define BRA_IA2AV_UNROLL 8
#endif
constexpr int kUnroll = BRA_IA2AV_UNROLL;   // positions in flight per thread

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

template <typename E>
__global__ void __launch_bounds__(kThreads, 1) ia2av_kernel(const __grid_constant__ IA2avArgs a) {
  extern __shared__ int64_t s_sc[];         // the P x P count matrix
  __shared__ int64_t s_rowtot[kA2avMaxP];
  __shared__ int64_t s_rowoff[kA2avMaxP];   // rank offsets in the concatenated send lists
  __shared__ int64_t s_cnt[kA2avMaxP];      // send_counts[i][j] of the current rank i
  __shared__ int64_t s_sd[kA2avMaxP];       // send_displs[i][j]
  __shared__ int64_t s_rd[kA2avMaxP];       // recv_displs[j][i]: where rank j puts rank i's part
  __shared__ int64_t s_range[2];            // this block's [lo, hi)
  const int P = a.P;
  const int nb = gridDim.x, b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // 1. the whole count matrix (one coalesced pass), its row totals, and the
  //    checks: negative counts, NULL buffers that would be used
  int bad = 0;
  for (int e = tid; e < P * P; e += kThreads) {
    const int64_t c = a.sc[e];
    s_sc[e] = c;
    bad |= c < 0;
  }
  __syncthreads();
  for (int r = warp; r < P; r += kWarps) {
    int64_t row = 0;
    for (int k = lane; k < P; k += 32) row += s_sc[r * P + k];
    row = warp_sum64(row);
    if (lane == 0) s_rowtot[r] = row;
  }
  for (int r = tid; r < P; r += kThreads) {
    int64_t row = 0, col = 0;
    for (int k = 0; k < P; ++k) {
      row += s_sc[r * P + k];
      col += s_sc[k * P + r];
    }
    if (row > 0 && a.idx[r] == nullptr) bad = 1;
    if (col > 0 && a.out[r] == nullptr) bad = 1;
  }
  if (__syncthreads_or(bad)) {
    if (b == 0 && tid == 0 && a.status) *a.status = BRA_ERR_INVALID;
    return;
  }
  if (warp == 0) {
    const int64_t v0 = lane < P ? s_rowtot[lane] : 0;
    const int64_t v1 = lane + 32 < P ? s_rowtot[lane + 32] : 0;
    int64_t o0, o1, N;
    warp_exscan64(v0, v1, lane, o0, o1, N);
    if (lane < P) s_rowoff[lane] = o0;
    if (lane + 32 < P) s_rowoff[lane + 32] = o1;
    if (lane == 0) {
      // even split of the N positions: the first N % nb blocks take one more
      const int64_t q = N / nb, rem = N % nb;
      s_range[0] = q * b + (b < rem ? b : rem);
      s_range[1] = s_range[0] + q + (b < rem ? 1 : 0);
    }
  }
  __syncthreads();
  const int64_t lo = s_range[0], hi = s_range[1];

  // 2. bookkeeping, entries (i, j) dealt round-robin over the blocks
  for (int64_t e = b + (int64_t)nb * tid; e < (int64_t)P * P; e += (int64_t)nb * kThreads) {
    const int i = (int)(e / P), j = (int)(e % P);
    int64_t sd = 0, rd = 0;
    for (int k = 0; k < j; ++k) sd += s_sc[i * P + k];
    for (int k = 0; k < i; ++k) rd += s_sc[k * P + j];
    a.sd[(int64_t)i * P + j] = sd;
    a.rc[(int64_t)j * P + i] = s_sc[i * P + j];
    a.rd[(int64_t)j * P + i] = rd;
  }

  // 3. the block's positions, rank by rank, destination by destination
  int oob = 0;
  for (int i = 0; i < P; ++i) {
    const int64_t off = s_rowoff[i], tot = s_rowtot[i];
    if (tot == 0 || off >= hi || off + tot <= lo) continue;   // uniform over the block
    const int64_t plo = lo > off ? lo - off : 0;              // this block's part of rank i
    const int64_t phi = hi - off < tot ? hi - off : tot;
    __syncthreads();   // the previous rank's tables are no longer read
    if (tid < P) {
      const int j = tid;
      s_cnt[j] = s_sc[i * P + j];
      int64_t sd = 0, rd = 0;
      for (int k = 0; k < j; ++k) sd += s_sc[i * P + k];
      for (int k = 0; k < i; ++k) rd += s_sc[k * P + j];
      s_sd[j] = sd;
      s_rd[j] = rd;
    }
    __syncthreads();
    const E* in = static_cast<const E*>(a.in[i]);
    const int64_t* idx = a.idx[i];
    const int64_t len = a.in_len[i];
    for (int j = 0; j < P; ++j) {
      const int64_t p0 = s_sd[j] > plo ? s_sd[j] : plo;
      const int64_t e0 = s_sd[j] + s_cnt[j];
      const int64_t p1 = e0 < phi ? e0 : phi;
      if (p0 >= p1) continue;
      E* dst = static_cast<E*>(a.out[j]);
      const int64_t shift = s_rd[j] - s_sd[j];   // out_j position = k + shift
      for (int64_t k0 = p0 + tid; k0 < p1; k0 += (int64_t)kThreads * kUnroll) {
        int64_t v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t k = k0 + (int64_t)u * kThreads;
          v[u] = k < p1 ? __ldg(idx + k) : -1;
        }
        E val[kUnroll];
        bool ok[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t k = k0 + (int64_t)u * kThreads;
          ok[u] = k < p1 && v[u] >= 0 && v[u] < len;
          if (k < p1 && !ok[u]) oob = 1;
          val[u] = ok[u] ? __ldg(in + v[u]) : E(0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (ok[u]) dst[k0 + (int64_t)u * kThreads + shift] = val[u];
      }
    }
  }
  if (__syncthreads_or(oob) && tid == 0 && a.status) atomicExch(a.status, (int32_t)BRA_ERR_INVALID);
}

// Per device: SM count and the shared memory a block may take.
struct IA2avDeviceInfo {
  bool ready = false;
  int sms = 0;
  int dyn_max = 0;
};

cudaError_t ia2av_device_info(IA2avDeviceInfo* out) {
  static std::mutex mu;
  static IA2avDeviceInfo info[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  IA2avDeviceInfo& di = info[dev & 63];
  if (!di.ready) {
    int sms = 0, optin = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
        cudaSuccess)
      return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, ia2av_kernel<uint8_t>)) != cudaSuccess) return e;
    di.dyn_max = optin - (int)fa.sharedSizeBytes;
    if ((e = cudaFuncSetAttribute(ia2av_kernel<uint8_t>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, di.dyn_max)) !=
        cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(ia2av_kernel<uint32_t>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, di.dyn_max)) !=
        cudaSuccess)
      return e;
    di.sms = sms > 0 ? sms : 1;
    di.ready = true;
  }
  *out = di;
  return cudaSuccess;
}

}  // namespace

int ia2av_launch_blocks(int64_t L) {
  IA2avDeviceInfo di;
  if (ia2av_device_info(&di) != cudaSuccess) return -1;
  return L < di.sms ? (int)L : di.sms;
}

cudaError_t launch_ia2av(const IA2avArgs& a, int blocks, cudaStream_t st) {
  IA2avDeviceInfo di;
  cudaError_t e = ia2av_device_info(&di);
  if (e != cudaSuccess) return e;
  if (blocks < 1 || (size_t)a.P * a.P * sizeof(int64_t) > (size_t)di.dyn_max)
    return cudaErrorInvalidConfiguration;
  const size_t smem = (size_t)a.P * a.P * sizeof(int64_t);   // at most 32 KiB
  if (a.esize == 4)
    ia2av_kernel<uint32_t><<<blocks, kThreads, smem, st>>>(a);
  else
    ia2av_kernel<uint8_t><<<blocks, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace bra
