// Row repacking for the workspace path of bmm_rs_a2a: operands whose rows are
// not 16-byte aligned (M/tp or H not a multiple of 8 elements, or a pointer
// only element-aligned) are copied, row by row, into caller-provided
// workspace with a pitch that is a multiple of 64 elements (128 bytes, so
// every row of a TMA box starts on an L2 line).  The tensor-core
// kernels then read the copies through ordinary 128-byte-swizzle TMA maps
// whose dimensions are the logical row lengths, so the padding is never
// read (TMA fills coordinates past a row's end with zeros).
//
// One warp copies one row at a time.  The source row starts at an even byte
// address; lanes load consecutive 32-bit words of it (coalesced, 128 bytes
// per warp instruction) and, when the row starts in the upper half of a word,
// join each word with its neighbour by a 16-bit funnel shift.  Only words
// that hold at least one byte of the row are read, so every load stays inside
// the 16-byte granules the row occupies (inside its allocation).  Stores are
// consecutive 32-bit words of the destination row; when the row length is odd
// the last word carries one padding element (zero), which lies inside the
// destination pitch.  Pure data movement: HBM-bound, 4 bytes read and 4 bytes
// written per element pair.
#include "bra_internal.h"

namespace bra {

namespace {

constexpr int kRThreads = 256;
constexpr int kRUnroll = 16;  // 32-bit words per lane per pass (2 KB per warp in flight)

__global__ void __launch_bounds__(kRThreads) repack_rows_kernel(const __grid_constant__ RepackArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kRThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kRThreads) >> 5;
  for (int64_t g = warp; g < a.total_rows; g += nwarps) {
    // the job holding row g: the last one whose first row is <= g
    int lo = 0, hi = a.njobs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.job[mid].row0 <= g) lo = mid;
      else hi = mid - 1;
    }
    const RepackJob& jb = a.job[lo];
    const int64_t row = g - jb.row0;
    const uintptr_t sa = reinterpret_cast<uintptr_t>(jb.src) + (uintptr_t)(row * jb.len * 2);
    uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(jb.dst) +
                                                row * (int64_t)jb.pitch * 2);
    const uintptr_t wa = sa & ~uintptr_t(3);          // word holding the first element
    const uint32_t* w0 = reinterpret_cast<const uint32_t*>(wa);
    const bool odd = (sa & 3) != 0;                   // first element in a word's upper half
    const uintptr_t end = sa + (uintptr_t)jb.len * 2; // one past the row's last byte
    const int64_t nsrc = (int64_t)((end - wa + 3) >> 2);   // words holding a byte of the row
    const int64_t nout = ((int64_t)jb.len + 1) >> 1;        // destination words
    for (int64_t base = 0; base < nout; base += 32 * kRUnroll) {
      uint32_t v[kRUnroll], nb[kRUnroll];
#pragma unroll
      for (int u = 0; u < kRUnroll; ++u) {
        const int64_t k = base + u * 32 + lane;
        v[u] = k < nsrc ? __ldg(w0 + k) : 0u;
      }
      if (odd) {
#pragma unroll
        for (int u = 0; u < kRUnroll; ++u) {
          const int64_t k1 = base + u * 32 + lane + 1;
          const uint32_t from_peer = __shfl_down_sync(0xffffffffu, v[u], 1);
          nb[u] = lane < 31 ? from_peer : (k1 < nsrc ? __ldg(w0 + k1) : 0u);
        }
#pragma unroll
        for (int u = 0; u < kRUnroll; ++u) v[u] = __funnelshift_r(v[u], nb[u], 16);
      }
#pragma unroll
      for (int u = 0; u < kRUnroll; ++u) {
        const int64_t k = base + u * 32 + lane;
        if (k < nout) {
          // an odd length leaves the upper half of the last word past the row
          uint32_t w = v[u];
          if ((jb.len & 1) && k == nout - 1) w &= 0xffffu;
          dst[k] = w;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_repack(const RepackArgs& a, cudaStream_t st) {
  if (a.total_rows <= 0 || a.njobs <= 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // 8 resident CTAs of 256 threads per SM; no more warps than rows
  const int64_t want = (a.total_rows + kRThreads / 32 - 1) / (kRThreads / 32);
  const int64_t full = (int64_t)sms * 8;
  const unsigned grid = (unsigned)(want < full ? want : full);
  repack_rows_kernel<<<grid, kRThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace bra
