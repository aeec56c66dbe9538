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
// Kernel shape: grid (parts, P); the `parts` CTAs of sender i split its n_i
// positions evenly.  Every CTA reads the whole count matrix first and rejects
// the call (nothing written) on a negative count or a NULL buffer that would
// be touched, so all CTAs take the same decision without talking to each
// other (the matrix is staged in shared memory with one coalesced pass).  In
// the copy, consecutive threads take consecutive positions: index loads and
// stores are coalesced, the gathers follow the index; each thread keeps four
// positions in flight (deeper unrolling measured no faster).  An index outside [0, in_len_i) is never dereferenced; its
// position is not delivered and the optional status word gets
// BRA_ERR_INVALID.  There are no waits.
#include <mutex>

#include "bra_internal.h"

namespace bra {

namespace {

constexpr int kThreads = 256;
#ifndef BRA_IA2AV_UNROLL
#define BRA_IA2AV_UNROLL 4
#endif
constexpr int kUnroll = BRA_IA2AV_UNROLL;   // positions in flight per thread

template <typename E>
__global__ void __launch_bounds__(kThreads) ia2av_kernel(const __grid_constant__ IA2avArgs a) {
  extern __shared__ int64_t s_sc[];       // the P x P count matrix
  __shared__ int64_t s_cnt[kA2avMaxP];   // send_counts[i][j]
  __shared__ int64_t s_sd[kA2avMaxP];    // send_displs[i][j]
  __shared__ int64_t s_rd[kA2avMaxP];    // recv_displs[j][i]: where rank j puts rank i's part
  const int P = a.P;
  const int i = blockIdx.y;
  const int part = blockIdx.x, parts = gridDim.x;
  const int tid = threadIdx.x;

  // 1. the whole count matrix, staged with one coalesced pass: negative
  //    counts, NULL buffers that would be used
  int bad = 0;
  for (int e = tid; e < P * P; e += kThreads) {
    s_sc[e] = a.sc[e];
    if (s_sc[e] < 0) bad = 1;
  }
  __syncthreads();
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
    if (i == 0 && part == 0 && tid == 0 && a.status) *a.status = BRA_ERR_INVALID;
    return;
  }

  // 2. rank i's row and the receivers' displacements for it
  if (tid < P) {
    s_cnt[tid] = s_sc[i * P + tid];
    int64_t run = 0;
    for (int k = 0; k < i; ++k) run += s_sc[k * P + tid];
    s_rd[tid] = run;
  }
  __syncthreads();
  if (tid == 0) {
    int64_t run = 0;
    for (int j = 0; j < P; ++j) {
      s_sd[j] = run;
      run += s_cnt[j];
    }
  }
  __syncthreads();
  const int64_t n = s_sd[P - 1] + s_cnt[P - 1];

  // 3. bookkeeping rows of rank i (one CTA per rank)
  if (part == 0 && tid < P) {
    const int j = tid;
    a.sd[i * P + j] = s_sd[j];
    a.rc[i * P + j] = s_sc[j * P + i];
    int64_t run = 0;
    for (int k = 0; k < j; ++k) run += s_sc[k * P + i];
    a.rd[i * P + j] = run;
  }

  // 4. this CTA's positions [lo, hi), destination by destination
  // even split: the first n % parts CTAs take one position more
  const int64_t q = n / parts, rem = n % parts;
  const int64_t lo = q * part + (part < rem ? part : rem);
  const int64_t hi = lo + q + (part < rem ? 1 : 0);
  const E* in = static_cast<const E*>(a.in[i]);
  const int64_t* idx = a.idx[i];
  const int64_t len = a.in_len[i];
  int oob = 0;
  for (int j = 0; j < P; ++j) {
    const int64_t p0 = s_sd[j] > lo ? s_sd[j] : lo;
    const int64_t e0 = s_sd[j] + s_cnt[j];
    const int64_t p1 = e0 < hi ? e0 : hi;
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
  if (__syncthreads_or(oob) && tid == 0 && a.status) atomicExch(a.status, (int32_t)BRA_ERR_INVALID);
}

}  // namespace

// CTAs per rank that fill the GPU once (resident CTAs / P), computed once per
// device and P: the occupancy query is a slow host call.
int ia2av_ctas_per_rank(int P) {
  if (P < 1 || P > kA2avMaxP) return 1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  static std::mutex mu;
  static int cache[64][kA2avMaxP + 1] = {};
  std::lock_guard<std::mutex> lk(mu);
  int& c = cache[dev & 63][P];
  if (c == 0) {
    int sms = 148, per_sm = 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t smem = (size_t)P * P * sizeof(int64_t);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ia2av_kernel<uint8_t>, kThreads,
                                                      smem) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    c = sms * per_sm / P;
    if (c < 1) c = 1;
  }
  return c;
}

cudaError_t launch_ia2av(const IA2avArgs& a, int ctas_per_rank, cudaStream_t st) {
  const dim3 grid((unsigned)ctas_per_rank, (unsigned)a.P);
  const size_t smem = (size_t)a.P * a.P * sizeof(int64_t);   // at most 32 KiB
  if (a.esize == 4)
    ia2av_kernel<uint32_t><<<grid, kThreads, smem, st>>>(a);
  else
    ia2av_kernel<uint8_t><<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace bra
