// Epilogue of the tensor-core kernels for outputs of any alignment
// (fused_tcu.cu, fused_tcr.cu, and fused_tc*.cu when an output or bias is
// not 16-byte aligned): one warp drains its 32 TMEM lanes of a 256-column
// fp32 accumulator, adds the sender's bias in fp32, rounds once and writes
// every element to its all-to-all destination (CANN guide
// "BatchMatMulReduceScatterAllToAll 原理、shape 约束与 aclnn 两段式调用",
// 功能说明与计算流程):
//   yShardType 0: y[j*tp + n/Hp][s*El+e, m%C, n%Hp]
//   yShardType 1: y[j*tp + (m%C)/Cp][s*El+e, (m%C)%Cp, n]      (j = m / C)
// A row's 64-column segment lands on one contiguous 128-byte run of its
// destination unless it crosses the end of H or (yShardType 0) a TP rank's
// chunk.  Such a run starts `delta` elements past a 16-byte boundary; the
// segment is staged in shared memory shifted by delta, so that every whole
// 16-byte chunk of the run is one aligned vector store and only the two
// partial chunks at its ends are written element by element.  Segments that
// cross a boundary are written element by element.
#pragma once

#include "tc_ptx.cuh"

namespace bra {
namespace tc {

template <typename T>
struct Elt;
template <>
struct Elt<__half> {
  static __device__ __forceinline__ float bias(const void* p, int64_t i) {
    return __half2float(static_cast<const __half*>(p)[i]);
  }
};
template <>
struct Elt<__nv_bfloat16> {
  static __device__ __forceinline__ float bias(const void* p, int64_t i) {
    return static_cast<const float*>(p)[i];
  }
};

// Staging per epilogue warp: 32 row buffers of 144 bytes (a 64-column
// segment of 16-bit outputs shifted by up to 7 elements; nine 16-byte
// chunks) plus the segment's yShardType-0 bias (fp32, 64 columns).
constexpr int kURowStride = 144;
constexpr int kUStageBytes = 32 * kURowStride + 64 * 4;

// Accumulator rows row0 .. row0+31 (row index in ep*C of Z_{s,e}), columns
// n0 .. n0+255, at TMEM address t_base (this warp's lane quarter).  P is a
// kernel parameter block with bias[], y[], s0, El, C, H, tp, type, has_bias
// and rows.  Per 64-column segment: phase 1, lane = row: bias in fp32, one
// rounding, pairs packed and staged shifted by the run's delta; phase 2,
// the runs' seven whole middle chunks with every lane a (row, chunk) pair,
// then each lane its own run's two end chunks (at most three aligned
// 8/4/2-byte stores each); phase 3: segments that cross a boundary, lanes on
// consecutive columns.
// kPrefetch: load the tile's bias up front and unroll the store passes
// (faster where the epilogue warps have the SM sub-partitions' issue slots
// and registers to themselves; the kernels whose loader warps share them
// pass false).
template <typename T, bool kPrefetch, typename P>
__device__ __forceinline__ void epilogue_rows_u(const P& p, uint32_t t_base, int row0, int sl,
                                                int e, int n0, uint8_t* stage, int lane) {
  constexpr int BN = 256;
  float* bias_stg = reinterpret_cast<float*>(stage + 32 * kURowStride);
  const int s = p.s0 + sl;
  const int Hp = p.H / p.tp;
  const int Cp = p.type == 1 ? p.C / p.tp : 1;
  const int m_own = row0 + lane;
  const bool own_ok = m_own < p.rows;
  const int t_own = (own_ok && p.type == 1) ? (m_own % p.C) / Cp : 0;
  // yShardType 1: the row picks the TP rank, hence the bias row.
  const void* brow = (p.has_bias && p.type == 1) ? p.bias[sl * p.tp + t_own] : nullptr;
  // This lane's row, once per tile: destination rank (without the column's
  // TP rank for yShardType 0) and element offset of its start.
  int d_own = 0;
  int64_t off_own = 0;
  if (own_ok) {
    const int j = m_own / p.C, cm = m_own - j * p.C;
    if (p.type == 0) {
      d_own = j * p.tp;
      off_own = ((int64_t)(s * p.El + e) * p.C + cm) * Hp;
    } else {
      d_own = j * p.tp + cm / Cp;
      off_own = ((int64_t)(s * p.El + e) * Cp + (cm % Cp)) * p.H;
    }
  }
  uint8_t* my_buf = stage + lane * kURowStride;
  // The bias is staged per segment and read by every row when it depends on
  // the column only: always for yShardType 0; for yShardType 1 when the
  // warp's rows all belong to one TP rank (row 0 of the warp is valid
  // whenever any is, since rows are consecutive).
  const int t_first = __shfl_sync(0xffffffffu, t_own, 0);
  const bool staged_bias =
      p.has_bias && (p.type == 0 || __all_sync(0xffffffffu, !own_ok || t_own == t_first));
  const void* brow_first = (p.has_bias && p.type == 1) ? p.bias[sl * p.tp + t_first] : nullptr;
  // the lane's eight bias values of the tile (columns lane + 32 i), loaded
  // together up front so that their latency is paid once per tile
  float bpre[BN / 32];
#pragma unroll
  for (int i = 0; i < BN / 32; ++i) {
    const int n = n0 + lane + 32 * i;
    float b = 0.f;
    if (kPrefetch && staged_bias && n < p.H) {
      if (p.type == 0) {
        const int t = n / Hp;
        b = Elt<T>::bias(p.bias[sl * p.tp + t], (int64_t)e * Hp + (n - t * Hp));
      } else {
        b = Elt<T>::bias(brow_first, (int64_t)e * p.H + n);
      }
    }
    bpre[i] = b;
  }
#pragma unroll 1
  for (int ch = 0; ch < BN / 64; ++ch) {
    const int nc = n0 + ch * 64;   // the segment's first column
    if (staged_bias) {
      float b0 = 0.f, b1 = 0.f;
      if (kPrefetch) {
        // the segment's two values of this lane, picked without indexing
        b0 = ch == 0 ? bpre[0] : ch == 1 ? bpre[2] : ch == 2 ? bpre[4] : bpre[6];
        b1 = ch == 0 ? bpre[1] : ch == 1 ? bpre[3] : ch == 2 ? bpre[5] : bpre[7];
      } else {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int n = nc + lane + 32 * half;
          float b = 0.f;
          if (n < p.H) {
            if (p.type == 0) {
              const int t = n / Hp;
              b = Elt<T>::bias(p.bias[sl * p.tp + t], (int64_t)e * Hp + (n - t * Hp));
            } else {
              b = Elt<T>::bias(brow_first, (int64_t)e * p.H + n);
            }
          }
          (half ? b1 : b0) = b;
        }
      }
      bias_stg[lane] = b0;
      bias_stg[lane + 32] = b1;
      __syncwarp();
    }
    uint32_t v[64];
    tmem_ld32(t_base + ch * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
    tmem_ld32(t_base + ch * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
    tmem_ld_wait();
    // the segment's destination run, when it is one
    bool fast = false;
    int delta = 0;
    uintptr_t abase = 0;
    if (own_ok && nc + 64 <= p.H) {
      int d = d_own;
      int64_t off = off_own + nc;
      bool one_run = true;
      if (p.type == 0) {
        const int t0 = nc / Hp;
        one_run = nc + 63 < (t0 + 1) * Hp;
        d = d_own + t0;
        off = off_own + (nc - t0 * Hp);
      }
      if (one_run) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(static_cast<uint16_t*>(p.y[d]) + off);
        delta = (int)((a & 15u) >> 1);
        abase = a - (a & 15u);
        fast = true;
      }
    }
    // phase 1: bias, round, pack (column 2i in the low half of w[i])
    if (staged_bias) {   // the segment's bias by 16-byte broadcast reads
#pragma unroll
      for (int i4 = 0; i4 < 16; ++i4) {
        const float4 b = reinterpret_cast<const float4*>(bias_stg)[i4];
        v[4 * i4 + 0] = __float_as_uint(__uint_as_float(v[4 * i4 + 0]) + b.x);
        v[4 * i4 + 1] = __float_as_uint(__uint_as_float(v[4 * i4 + 1]) + b.y);
        v[4 * i4 + 2] = __float_as_uint(__uint_as_float(v[4 * i4 + 2]) + b.z);
        v[4 * i4 + 3] = __float_as_uint(__uint_as_float(v[4 * i4 + 3]) + b.w);
      }
    }
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float f0 = __uint_as_float(v[2 * i]), f1 = __uint_as_float(v[2 * i + 1]);
      if (p.has_bias && !staged_bias) {
        if (own_ok) {
          const int n = nc + 2 * i;
          if (n < p.H) f0 += Elt<T>::bias(brow, (int64_t)e * p.H + n);
          if (n + 1 < p.H) f1 += Elt<T>::bias(brow, (int64_t)e * p.H + n + 1);
        }
      }
      w[i] = Out<T>::pack(f0, f1);   // one paired RNE conversion: f0 low, f1 high
    }
    // stage: buffer element k holds column k - delta (delta = 0 off the fast
    // path).  Word q + i of the row buffer (q = delta / 2) joins w[i-1] and
    // w[i] by a funnel shift of 16 bits for an odd delta and of 32 (w[i]
    // alone) for an even one, so every lane runs the same instructions.
    uint32_t* bw = reinterpret_cast<uint32_t*>(my_buf);
    const int q = delta >> 1;
    const uint32_t sh = (delta & 1) ? 16u : 32u;
    bw[q] = __funnelshift_rc(0u, w[0], sh);
#pragma unroll
    for (int i = 1; i < 32; ++i) bw[q + i] = __funnelshift_rc(w[i - 1], w[i], sh);
    bw[q + 32] = __funnelshift_rc(w[31], 0u, sh);
    __syncwarp();
    // phase 2a: a run covers buffer bytes [2 delta, 2 delta + 128), so its
    // chunks 1..7 are always whole 16-byte vectors: 32 rows x 7 chunks, seven
    // passes of the warp.  A row's metadata travels as one word: its run's
    // 16-byte aligned start with delta in the low bits (0: off the fast path).
    const uint64_t meta = fast ? ((uint64_t)abase | (uint64_t)delta) : 0ull;
#pragma unroll(kPrefetch ? 7 : 1)
    for (int pass = 0; pass < 7; ++pass) {
      const int idx = pass * 32 + lane;
      const int rr = idx / 7, k = 1 + idx - 7 * rr;
      const uint32_t mlo = __shfl_sync(0xffffffffu, (uint32_t)meta, rr);
      const uint32_t mhi = __shfl_sync(0xffffffffu, (uint32_t)(meta >> 32), rr);
      const uint64_t m = ((uint64_t)mhi << 32) | mlo;
      if (m != 0) {
        const uint4 val = *reinterpret_cast<const uint4*>(stage + rr * kURowStride + 16 * k);
        *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(m & ~(uint64_t)15) + 16 * k) = val;
      }
    }
    // phase 2b: the end chunks of the lane's own run: chunk 0 (whole when
    // delta is 0, else its bytes [2 delta, 16)) and chunk 8 (its bytes
    // [0, 2 delta) when delta > 0), with at most three aligned 8/4/2-byte
    // stores each.
    if (fast) {
      uint8_t* ab = reinterpret_cast<uint8_t*>(abase);
      const int lo = 2 * delta;
      const uint4 v0 = *reinterpret_cast<const uint4*>(my_buf);
      if (lo == 0) {
        *reinterpret_cast<uint4*>(ab) = v0;
      } else {
        auto w0 = [&](int i) { return i == 0 ? v0.x : i == 1 ? v0.y : i == 2 ? v0.z : v0.w; };
        int b = lo;                                 // head: bytes [lo, 16)
        if (b & 2) {
          *reinterpret_cast<uint16_t*>(ab + b) = (uint16_t)(w0(b >> 2) >> 16);
          b += 2;
        }
        if (b & 4) {
          *reinterpret_cast<uint32_t*>(ab + b) = w0(b >> 2);
          b += 4;
        }
        if (b & 8) *reinterpret_cast<uint2*>(ab + b) = make_uint2(v0.z, v0.w);
        const uint4 v8 = *reinterpret_cast<const uint4*>(my_buf + 128);
        auto w8 = [&](int i) { return i == 0 ? v8.x : i == 1 ? v8.y : i == 2 ? v8.z : v8.w; };
        uint8_t* tl = ab + 128;                     // tail: bytes [0, lo)
        if (lo & 8) *reinterpret_cast<uint2*>(tl) = make_uint2(v8.x, v8.y);
        const int b4 = lo & 8;
        if (lo & 4) *reinterpret_cast<uint32_t*>(tl + b4) = w8(b4 >> 2);
        const int b2 = lo & 12;
        if (lo & 2) *reinterpret_cast<uint16_t*>(tl + b2) = (uint16_t)w8(b2 >> 2);
      }
    }
    // phase 3: valid rows off the fast path, element by element
    uint32_t slow = __ballot_sync(0xffffffffu, own_ok && !fast);
    const int n = nc + lane;
    while (slow) {
      const int rr = __ffs(slow) - 1;
      slow &= slow - 1;
      const int d0 = __shfl_sync(0xffffffffu, d_own, rr);
      const int64_t o0 = __shfl_sync(0xffffffffu, off_own, rr);
      const uint16_t* rb = reinterpret_cast<const uint16_t*>(stage + rr * kURowStride);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int nn = n + 32 * half;
        if (nn < p.H) {
          const int t_n = p.type == 0 ? nn / Hp : 0;
          const int h_n = nn - t_n * (p.type == 0 ? Hp : 0);
          static_cast<uint16_t*>(p.y[d0 + t_n])[o0 + h_n] = rb[lane + 32 * half];
        }
      }
    }
    __syncwarp();
  }
}

}  // namespace tc
}  // namespace bra
