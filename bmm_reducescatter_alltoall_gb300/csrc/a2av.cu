// all_to_all_v among P virtual ranks resident on one GPU.
//
// Semantics ("LowerL2TensorCollectives Pass", 行为 / ABI; addressing as in
// the meta ncclx alltoallv of "vccl alltoallv dev log", 5. ref): rank i sends
// send_counts[i][j] elements to rank j; displacements are exclusive prefix
// sums in element units, over destinations for the sender and over sources
// for the receiver.
//
// One launch, grid (ctas_per_rank, P).  Every CTA of source rank i:
//   1. stages the whole P x P count matrix in shared memory (P <= 64) and
//      rejects the call if any count is negative (every CTA sees the same
//      matrix, so all of them take the same decision without a grid sync);
//   2. warp-scans row i (its send displacements) and, per column j, the
//      counts of sources k < i (its receive displacement at rank j);
//   3. CTA 0 of rank i writes row i of send_displs and column i of
//      recv_counts / recv_displs;
//   4. copies: rank i's send buffer is split into B = CalAllToAllVBlocks(P, L)
//      equal element ranges ("blocks"); CTA c handles blocks c, c + C, ...
//      Each block range is cut at the destination boundaries and every piece
//      is a byte copy done by the whole CTA with 16-byte stores aligned on the
//      destination; when source and destination differ in alignment the
//      16-byte source words are funnel-shifted into place (int8 can be off by
//      any byte, fp32 by whole words).  Head and tail bytes are single-byte
//      copies.
// No CTA waits on another, so there is nothing that can hang.
#include <cstdint>

#include "bra_internal.h"

namespace bra {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Exclusive scan of 64 values held as (lane, lane + 32) by one warp.
__device__ __forceinline__ void warp_exscan64(int64_t v0, int64_t v1, int lane,
                                              int64_t& ex0, int64_t& ex1,
                                              int64_t& total) {
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

// Output word q of the 16 destination bytes = source bytes [4q + delta, ...),
// taken from the 32 source bytes (a, b) that start at an aligned address.
template <int Q>
__device__ __forceinline__ uint4 realign(const uint4& a, const uint4& b, uint32_t r) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint4 o;
  o.x = __funnelshift_r(w[Q + 0], w[Q + 1], r);
  o.y = __funnelshift_r(w[Q + 1], w[Q + 2], r);
  o.z = __funnelshift_r(w[Q + 2], w[Q + 3], r);
  o.w = __funnelshift_r(w[Q + 3], w[Q + 4], r);
  return o;
}

constexpr int kUnroll = 4;

__device__ __forceinline__ void copy_vec_aligned(uint4* __restrict__ d,
                                                 const uint4* __restrict__ s,
                                                 int64_t nvec) {
  const int64_t step = blockDim.x;
  int64_t v = threadIdx.x;
  for (; v + (kUnroll - 1) * step < nvec; v += kUnroll * step) {
    uint4 a[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) a[u] = __ldg(s + v + u * step);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) d[v + u * step] = a[u];
  }
  for (; v < nvec; v += step) d[v] = __ldg(s + v);
}

// s points at the aligned 16-byte word holding the first source byte; the
// last word read, s[nvec], holds at least one needed byte, so every load
// stays inside a 16-byte granule the source buffer occupies.
template <int Q>
__device__ __forceinline__ void copy_vec_shifted(uint4* __restrict__ d,
                                                 const uint4* __restrict__ s,
                                                 int64_t nvec, uint32_t r) {
  const int64_t step = blockDim.x;
  int64_t v = threadIdx.x;
  for (; v + (kUnroll - 1) * step < nvec; v += kUnroll * step) {
    uint4 a[kUnroll], b[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      a[u] = __ldg(s + v + u * step);
      b[u] = __ldg(s + v + u * step + 1);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) d[v + u * step] = realign<Q>(a[u], b[u], r);
  }
  for (; v < nvec; v += step) d[v] = realign<Q>(__ldg(s + v), __ldg(s + v + 1), r);
}

// Copy n bytes with the whole CTA.
__device__ void cta_copy_bytes(char* __restrict__ dst, const char* __restrict__ src,
                               int64_t n) {
  const int tid = threadIdx.x;
  int64_t head = (16 - (int64_t)((uintptr_t)dst & 15)) & 15;
  if (head > n) head = n;
  if (tid < head) dst[tid] = src[tid];
  dst += head;
  src += head;
  n -= head;
  const int64_t nvec = n >> 4;
  const int tail = (int)(n & 15);
  const uint32_t delta = (uint32_t)((uintptr_t)src & 15);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  if (nvec > 0) {
    if (delta == 0) {
      copy_vec_aligned(d4, reinterpret_cast<const uint4*>(src), nvec);
    } else {
      const uint4* s4 = reinterpret_cast<const uint4*>(src - delta);
      const uint32_t r = (delta & 3u) * 8u;
      switch (delta >> 2) {
        case 0: copy_vec_shifted<0>(d4, s4, nvec, r); break;
        case 1: copy_vec_shifted<1>(d4, s4, nvec, r); break;
        case 2: copy_vec_shifted<2>(d4, s4, nvec, r); break;
        default: copy_vec_shifted<3>(d4, s4, nvec, r); break;
      }
    }
  }
  if (tid < tail) dst[nvec * 16 + tid] = src[nvec * 16 + tid];
}

// Start of equal range b of B over n elements (ranges differ by at most one).
__device__ __forceinline__ int64_t split_point(int64_t n, int64_t B, int64_t b) {
  const int64_t q = n / B, rem = n % B;
  return q * b + (b < rem ? b : rem);
}

__global__ void __launch_bounds__(kA2avThreads)
a2av_kernel(const __grid_constant__ A2avArgs a) {
  __shared__ int64_t s_sc[kA2avMaxP * kA2avMaxP];
  __shared__ int64_t s_sd[kA2avMaxP];    // send displacement of rank i to j
  __shared__ int64_t s_rd[kA2avMaxP];    // receive displacement of i at j
  __shared__ int64_t s_tot[kA2avMaxP];   // elements rank j receives
  __shared__ int s_bad;

  const int P = a.P;
  const int i = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;

  if (tid == 0) s_bad = 0;
  __syncthreads();
  for (int k = tid; k < P * P; k += blockDim.x) {
    const int64_t v = a.sc[k];
    s_sc[k] = v;
    if (v < 0) s_bad = 1;
  }
  __syncthreads();

  if (warp == 0) {
    const int64_t v0 = lane < P ? s_sc[i * P + lane] : 0;
    const int64_t v1 = lane + 32 < P ? s_sc[i * P + lane + 32] : 0;
    int64_t e0, e1, tot;
    warp_exscan64(v0, v1, lane, e0, e1, tot);
    if (lane < P) s_sd[lane] = e0;
    if (lane + 32 < P) s_sd[lane + 32] = e1;
  }
  for (int j = warp; j < P; j += nwarps) {
    const int64_t v0 = lane < P ? s_sc[lane * P + j] : 0;
    const int64_t v1 = lane + 32 < P ? s_sc[(lane + 32) * P + j] : 0;
    int64_t e0, e1, tot;
    warp_exscan64(v0, v1, lane, e0, e1, tot);
    const int64_t at_i = __shfl_sync(kFull, i < 32 ? e0 : e1, i & 31);
    if (lane == 0) {
      s_rd[j] = at_i;
      s_tot[j] = tot;
    }
  }
  __syncthreads();

  if (tid == 0 && a.check_cap && !s_bad) {
    for (int j = 0; j < P; ++j)
      if (s_tot[j] > a.cap[j]) s_bad = 1;
  }
  __syncthreads();
  const bool bad = s_bad != 0;
  if (a.status && blockIdx.x == 0 && i == 0 && tid == 0)
    *a.status = bad ? BRA_ERR_INVALID : BRA_OK;
  if (bad) return;

  if (blockIdx.x == 0) {
    for (int j = tid; j < P; j += blockDim.x) {
      a.sd[(int64_t)i * P + j] = s_sd[j];
      a.rc[(int64_t)j * P + i] = s_sc[i * P + j];
      a.rd[(int64_t)j * P + i] = s_rd[j];
    }
  }

  const int64_t total = s_sd[P - 1] + s_sc[i * P + P - 1];
  const int64_t es = a.esize;
  const char* src = static_cast<const char*>(a.in[i]);
  for (int64_t b = blockIdx.x; b < a.B; b += gridDim.x) {
    const int64_t lo = split_point(total, a.B, b), hi = split_point(total, a.B, b + 1);
    if (lo >= hi) continue;
    for (int j = 0; j < P; ++j) {
      const int64_t seg_lo = s_sd[j], seg_hi = seg_lo + s_sc[i * P + j];
      const int64_t c0 = lo > seg_lo ? lo : seg_lo;
      const int64_t c1 = hi < seg_hi ? hi : seg_hi;
      if (c0 >= c1) continue;
      char* dst = static_cast<char*>(a.out[j]) + (s_rd[j] + (c0 - seg_lo)) * es;
      cta_copy_bytes(dst, src + c0 * es, (c1 - c0) * es);
    }
  }
}

__global__ void l2_flush_kernel(uint4* __restrict__ buf, size_t nvec) {
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x; k < nvec;
       k += (size_t)gridDim.x * blockDim.x)
    buf[k] = z;
}

__global__ void l2_flush_tail_kernel(char* __restrict__ buf, size_t n) {
  const size_t k = threadIdx.x;
  if (k < n) buf[k] = 0;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n > 0 ? n : 148;
}

}  // namespace

int a2av_ctas_per_rank(int P, int B) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, a2av_kernel, kA2avThreads, 0) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const long long resident = (long long)per_sm * device_sm_count();
  long long c = (resident + P - 1) / P;
  if (c < 1) c = 1;
  if (c > B) c = B;
  return (int)c;
}

cudaError_t launch_a2av(const A2avArgs& a, int ctas_per_rank, cudaStream_t st) {
  dim3 grid(ctas_per_rank, a.P);
  a2av_kernel<<<grid, kA2avThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_l2_flush(void* buf, size_t bytes, cudaStream_t st) {
  const size_t nvec = bytes / 16;
  const size_t tail = bytes - nvec * 16;
  if (nvec) {
    const int blocks = 4 * device_sm_count();
    l2_flush_kernel<<<blocks, 512, 0, st>>>(static_cast<uint4*>(buf), nvec);
  }
  if (tail) l2_flush_tail_kernel<<<1, 32, 0, st>>>(static_cast<char*>(buf) + nvec * 16, tail);
  return cudaGetLastError();
}

}  // namespace bra
