// Generic fused BMM -> TP ReduceScatter -> bias Add -> EP AllToAll kernel.
//
// Used for shapes the tensor-core kernel cannot take (row strides or
// pointers not 16-byte aligned, e.g. M/tp = 6 or H = 4 in the 8-rank example
// of the CANN guide, section 完整调用示例) and as an independent cross-check.
// Any size and alignment; scalar loads with bounds checks.
//
// Per output tile (64 x 64 of Z_{s,e}, s the source EP rank, e the local
// expert), the contraction runs over the tp shards t' = 0..tp-1 in order and,
// inside each, over k ascending, one fp32 FMA chain per output element; the
// reduce-scatter is this sum.  The epilogue adds the sender's bias in fp32,
// rounds once to the output dtype and stores every element at its all-to-all
// destination:
//   yShardType 0: row m = j*C + c, col n = t*Hp + h -> y[j*tp+t][s*El+e, c, h]
//   yShardType 1: row m = j*C + t*Cp + c, col h     -> y[j*tp+t][s*El+e, c, h]
// (CANN guide, 功能说明与计算流程 and 参数说明 yShardType).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>
#include <memory>

#include "bra_internal.h"

namespace bra {
namespace {

constexpr int kTile = 64, kTk = 16, kThreads = 256;

struct SimtParams {
  const void* x[kChunkRanks];
  const void* w[kChunkRanks];
  const void* bias[kChunkRanks];
  void* y[kMaxRanks];
  int ep, tp, El, C, Kp, H, type, has_bias;
  int wt;       // weight stored transposed: (El, H, Kp)
  int s0;       // first source EP rank of this launch
  int rows;     // ep * C
  int m_tiles;
};

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// grid: x = n tiles, y = m tiles (grid-stride), z = (s - s0) * El + e
template <typename T, typename BT>
__global__ void __launch_bounds__(kThreads)
fused_simt_kernel(const __grid_constant__ SimtParams p) {
  __shared__ float As[kTk][kTile + 4];
  __shared__ float Bs[kTk][kTile + 4];
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  const int sl = blockIdx.z / p.El, e = blockIdx.z % p.El, s = p.s0 + sl;
  const int n0 = blockIdx.x * kTile;
  const int Hp = p.H / p.tp, Cp = p.C / p.tp;
  const int64_t x_e = (int64_t)e * p.rows * p.Kp, w_e = (int64_t)e * p.Kp * p.H;

  for (int mt = blockIdx.y; mt < p.m_tiles; mt += gridDim.y) {
    const int m0 = mt * kTile;
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;

    for (int t = 0; t < p.tp; ++t) {
      const T* X = static_cast<const T*>(p.x[sl * p.tp + t]) + x_e;
      const T* W = static_cast<const T*>(p.w[sl * p.tp + t]) + w_e;
      for (int k0 = 0; k0 < p.Kp; k0 += kTk) {
#pragma unroll
        for (int q = 0; q < (kTile * kTk) / kThreads; ++q) {
          const int idx = tid + q * kThreads;
          const int am = idx / kTk, ak = idx % kTk;
          const int gm = m0 + am, gk = k0 + ak;
          As[ak][am] = (gm < p.rows && gk < p.Kp) ? to_f<T>(X[(int64_t)gm * p.Kp + gk]) : 0.f;
          const int bk = idx / kTile, bn = idx % kTile;
          const int gk2 = k0 + bk, gn = n0 + bn;
          const int64_t widx = p.wt ? (int64_t)gn * p.Kp + gk2 : (int64_t)gk2 * p.H + gn;
          Bs[bk][bn] = (gk2 < p.Kp && gn < p.H) ? to_f<T>(W[widx]) : 0.f;
        }
        __syncthreads();
        const int kn = min(kTk, p.Kp - k0);
        for (int k = 0; k < kn; ++k) {
          float av[4], bv[4];
#pragma unroll
          for (int a = 0; a < 4; ++a) av[a] = As[k][ty * 4 + a];
#pragma unroll
          for (int b = 0; b < 4; ++b) bv[b] = Bs[k][tx * 4 + b];
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(av[a], bv[b], acc[a][b]);
        }
        __syncthreads();
      }
    }

#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int m = m0 + ty * 4 + a;
      if (m >= p.rows) continue;
      const int j = m / p.C, cm = m % p.C;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int n = n0 + tx * 4 + b;
        if (n >= p.H) continue;
        int t, dst_row, col, bcol, Wd;
        if (p.type == 0) {
          t = n / Hp;
          dst_row = cm;
          col = n % Hp;
          bcol = col;
          Wd = Hp;
        } else {
          t = cm / Cp;
          dst_row = cm % Cp;
          col = n;
          bcol = n;
          Wd = p.H;
        }
        const int rows_d = p.type == 0 ? p.C : Cp;
        float v = acc[a][b];
        if (p.has_bias) {
          const BT* bp = static_cast<const BT*>(p.bias[sl * p.tp + t]);
          v += to_f<BT>(bp[(int64_t)e * Wd + bcol]);
        }
        T* yd = static_cast<T*>(p.y[j * p.tp + t]);
        const int64_t off = ((int64_t)(s * p.El + e) * rows_d + dst_row) * Wd + col;
        yd[off] = from_f<T>(v);
      }
    }
  }
}

}  // namespace

cudaError_t launch_fused_simt(const FusedProblem& f, cudaStream_t st) {
  std::unique_ptr<SimtParams> p(new SimtParams);
  std::memset(p.get(), 0, sizeof(SimtParams));
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
  p->wt = f.wt;
  p->rows = f.ep * f.C;
  p->m_tiles = (p->rows + kTile - 1) / kTile;
  const int s_per_launch = kChunkRanks / f.tp > 0 ? kChunkRanks / f.tp : 1;
  for (int s0 = 0; s0 < f.ep; s0 += s_per_launch) {
    const int s1 = s0 + s_per_launch < f.ep ? s0 + s_per_launch : f.ep;
    p->s0 = s0;
    for (int r = 0; r < (s1 - s0) * f.tp; ++r) {
      p->x[r] = f.x[s0 * f.tp + r];
      p->w[r] = f.w[s0 * f.tp + r];
      p->bias[r] = f.bias ? f.bias[s0 * f.tp + r] : nullptr;
    }
    dim3 grid((f.H + kTile - 1) / kTile, p->m_tiles < 65535 ? p->m_tiles : 65535,
              (s1 - s0) * f.El);
    if (f.dtype == BRA_FP16)
      fused_simt_kernel<__half, __half><<<grid, kThreads, 0, st>>>(*p);
    else
      fused_simt_kernel<__nv_bfloat16, float><<<grid, kThreads, 0, st>>>(*p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace bra
