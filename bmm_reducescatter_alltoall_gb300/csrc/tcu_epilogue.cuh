// Epilogue of the tensor-core kernels for rows of any alignment
// (fused_tcu.cu, fused_tcr.cu): one warp drains its 32 TMEM lanes of a
// 256-column fp32 accumulator, adds the sender's bias in fp32, rounds once
// and writes every element to its all-to-all destination with 2-byte stores
// (CANN guide "BatchMatMulReduceScatterAllToAll 原理、shape 约束与 aclnn
// 两段式调用", 功能说明与计算流程):
//   yShardType 0: y[j*tp + n/Hp][s*El+e, m%C, n%Hp]
//   yShardType 1: y[j*tp + (m%C)/Cp][s*El+e, (m%C)%Cp, n]      (j = m / C)
// Rows of any alignment and type-0 chunks that straddle a TP rank are fine.
#pragma once

#include "tc_ptx.cuh"

namespace bra {
namespace tc {

template <typename T>
struct Elt;
template <>
struct Elt<__half> {
  static __device__ __forceinline__ uint16_t cvt(float v) {
    return __half_as_ushort(__float2half_rn(v));
  }
  static __device__ __forceinline__ float bias(const void* p, int64_t i) {
    return __half2float(static_cast<const __half*>(p)[i]);
  }
};
template <>
struct Elt<__nv_bfloat16> {
  static __device__ __forceinline__ uint16_t cvt(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
  static __device__ __forceinline__ float bias(const void* p, int64_t i) {
    return static_cast<const float*>(p)[i];
  }
};

// Staging per epilogue warp: 32 rows x 32 rounded 16-bit outputs (64 bytes,
// rows 68 bytes apart so row-per-lane writes and per-row reads avoid bank
// conflicts) plus the tile's yShardType-0 bias (fp32, 256 columns).
constexpr int kURowStride = 68;
constexpr int kUStageBytes = 32 * kURowStride + 256 * 4;

// Accumulator rows row0 .. row0+31 (row index in ep*C of Z_{s,e}), columns
// n0 .. n0+255, at TMEM address t_base (this warp's lane quarter).  P is a
// kernel parameter block with bias[], y[], s0, El, C, H, tp, type, has_bias
// and rows.  Phase 1: lane = row; bias in fp32, one rounding, staged.
// Phase 2: row by row, lanes on consecutive columns; a row's destination is
// computed once by its own lane and broadcast.
template <typename T, typename P>
__device__ __forceinline__ void epilogue_rows_u(const P& p, uint32_t t_base, int row0, int sl,
                                                int e, int n0, uint8_t* stage, int lane) {
  constexpr int BN = 256;
  uint16_t* stg = reinterpret_cast<uint16_t*>(stage);
  float* bias_stg = reinterpret_cast<float*>(stage + 32 * kURowStride);
  const int s = p.s0 + sl;
  const int Hp = p.H / p.tp;
  const int Cp = p.type == 1 ? p.C / p.tp : 1;
  // yShardType 0: the bias depends on the column only.
  if (p.has_bias && p.type == 0) {
    for (int c = lane; c < BN; c += 32) {
      const int n = n0 + c;
      float b = 0.f;
      if (n < p.H) {
        const int t = n / Hp;
        b = Elt<T>::bias(p.bias[sl * p.tp + t], (int64_t)e * Hp + (n - t * Hp));
      }
      bias_stg[c] = b;
    }
    __syncwarp();
  }
  const int m_own = row0 + lane;
  const int t_own = (m_own < p.rows && p.type == 1) ? (m_own % p.C) / Cp : 0;
  // yShardType 1: the row picks the TP rank, hence the bias row.
  const void* brow = (p.has_bias && p.type == 1) ? p.bias[sl * p.tp + t_own] : nullptr;
  // This lane's row, once per tile: destination rank (without the column's
  // TP rank for yShardType 0) and element offset of its start.
  int d_own = 0;
  int64_t off_own = 0;
  if (m_own < p.rows) {
    const int j = m_own / p.C, cm = m_own - j * p.C;
    if (p.type == 0) {
      d_own = j * p.tp;
      off_own = ((int64_t)(s * p.El + e) * p.C + cm) * Hp;
    } else {
      d_own = j * p.tp + cm / Cp;
      off_own = ((int64_t)(s * p.El + e) * Cp + (cm % Cp)) * p.H;
    }
  }
#pragma unroll 1
  for (int ch = 0; ch < BN / 32; ++ch) {
    uint32_t v[32];
    tmem_ld32(t_base + ch * 32, v);
    tmem_ld_wait();
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      float f = __uint_as_float(v[c]);
      const int n = n0 + ch * 32 + c;
      if (p.has_bias) {
        if (p.type == 0)
          f += bias_stg[ch * 32 + c];
        else if (m_own < p.rows && n < p.H)
          f += Elt<T>::bias(brow, (int64_t)e * p.H + n);
      }
      stg[lane * (kURowStride / 2) + c] = Elt<T>::cvt(f);
    }
    __syncwarp();
    const int n = n0 + ch * 32 + lane;
    const int t_n = p.type == 0 ? n / Hp : 0;
    const int h_n = n - t_n * (p.type == 0 ? Hp : 0);
#pragma unroll 1
    for (int rr = 0; rr < 32; ++rr) {
      if (row0 + rr >= p.rows) break;
      const int d = __shfl_sync(0xffffffffu, d_own, rr) + t_n;
      const int64_t off = __shfl_sync(0xffffffffu, off_own, rr) + h_n;
      if (n < p.H) static_cast<uint16_t*>(p.y[d])[off] = stg[rr * (kURowStride / 2) + lane];
    }
    __syncwarp();
  }
}

}  // namespace tc
}  // namespace bra
