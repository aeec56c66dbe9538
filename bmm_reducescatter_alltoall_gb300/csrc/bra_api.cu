// Host entry points of libbmmrsa2a.so: argument validation, variant choice
// and launches.  Every rule cited here is stated in include/bmm_rs_a2a.h.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "bra_internal.h"

namespace {

constexpr int64_t kInt32Max = 2147483647LL;

bool world_size_ok(int64_t v) {
  return v == 1 || v == 2 || v == 4 || v == 8 || v == 16 || v == 32;
}

// Range rules of the CANN guide, section 数据关系与取值范围说明, and the
// attribute checks of section op_api 层 (CheckAttr / CheckShapeRange).
int check_fused_attrs(int64_t ep, int64_t tp, int64_t E, int64_t C, int64_t M,
                      int64_t H, int64_t type) {
  if (!world_size_ok(ep) || !world_size_ok(tp)) return BRA_ERR_INVALID;
  if (type != 0 && type != 1) return BRA_ERR_INVALID;
  if (E < 2 || E > 512 || E % ep != 0) return BRA_ERR_INVALID;
  if (E / ep < 1 || E / ep > 32) return BRA_ERR_INVALID;
  if (H < 1 || H > 65535) return BRA_ERR_INVALID;
  if (M % tp != 0 || M / tp < 1 || M / tp > 65535) return BRA_ERR_INVALID;
  if (C <= 0) return BRA_ERR_INVALID;
  if (type == 0 && H % tp != 0) return BRA_ERR_INVALID;
  if (type == 1 && C % tp != 0) return BRA_ERR_INVALID;
  return BRA_OK;
}

struct Range {
  uintptr_t lo, hi;
  bool out;
};

void tensor_ranges(const bra::FusedProblem& p, std::vector<Range>* all);
int apply_pitches(const bra_fused_options* opts, bra::FusedProblem* p);

// Validation in the order of CheckParams: null pointers, dtype, attributes,
// shapes; then the aliasing rule.  On success fills `prob`.
int validate_fused(const void* const x[], const void* const weight[],
                   const void* const bias[], int64_t ep, int64_t tp, int64_t E,
                   int64_t C, int64_t M, int64_t H, int64_t type, int dtype,
                   void* const out[], const bra_fused_options* opts,
                   bra::FusedProblem* prob) {
  if (!x || !weight || !out) return BRA_ERR_NULLPTR;
  if (dtype != BRA_FP16 && dtype != BRA_BF16) return BRA_ERR_INVALID;
  if (opts) {
    if (opts->x_pitch < 0 || opts->w_pitch < 0) return BRA_ERR_INVALID;
    if (opts->variant != BRA_VARIANT_AUTO && opts->variant != BRA_VARIANT_TC &&
        opts->variant != BRA_VARIANT_TC2 && opts->variant != BRA_VARIANT_SIMT &&
        opts->variant != BRA_VARIANT_TCU && opts->variant != BRA_VARIANT_TCR &&
        opts->variant != BRA_VARIANT_PACKED)
      return BRA_ERR_INVALID;
    if (opts->workspace_bytes < 0) return BRA_ERR_INVALID;
    if (!opts->workspace && opts->workspace_bytes != 0) return BRA_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(opts->workspace) & 255u) return BRA_ERR_INVALID;
  }
  int rc = check_fused_attrs(ep, tp, E, C, M, H, type);
  if (rc != BRA_OK) return rc;
  const int64_t P = ep * tp;
  for (int64_t r = 0; r < P; ++r)
    if (!x[r] || !weight[r] || !out[r]) return BRA_ERR_NULLPTR;
  int nb = 0;
  if (bias)
    for (int64_t r = 0; r < P; ++r) nb += bias[r] != nullptr;
  if (nb != 0 && nb != P) return BRA_ERR_INVALID;
  if (ep * C >= (int64_t(1) << 31)) return BRA_ERR_UNSUPPORTED;

  const int64_t El = E / ep, Kp = M / tp;
  prob->x = x;
  prob->w = weight;
  prob->bias = nb ? bias : nullptr;
  prob->y = out;
  prob->ep = (int)ep;
  prob->tp = (int)tp;
  prob->El = (int)El;
  prob->C = (int)C;
  prob->Kp = (int)Kp;
  prob->H = (int)H;
  prob->type = (int)type;
  prob->dtype = dtype;
  prob->wt = (opts && opts->transpose_weight) ? 1 : 0;
  prob->status = opts ? opts->status : nullptr;
  prob->xp = (int)Kp;
  prob->wp = prob->wt ? (int)Kp : (int)H;
  rc = apply_pitches(opts, prob);
  if (rc != BRA_OK) return rc;
  // Outputs may overlap nothing.  Sorted by start, a pair (a before b)
  // overlaps iff b.lo < a.hi; track the largest end of every earlier range
  // and of every earlier output.
  std::vector<Range> all;
  all.reserve(4 * P);
  tensor_ranges(*prob, &all);
  std::sort(all.begin(), all.end(),
            [](const Range& a, const Range& b) { return a.lo < b.lo; });
  uintptr_t max_hi_all = 0, max_hi_out = 0;
  for (const Range& a : all) {
    if (a.out ? a.lo < max_hi_all : a.lo < max_hi_out) return BRA_ERR_INVALID;
    max_hi_all = std::max(max_hi_all, a.hi);
    if (a.out) max_hi_out = std::max(max_hi_out, a.hi);
  }
  return BRA_OK;
}

// Caller pitches (elements; 0 = dense): each at least its row length.
int apply_pitches(const bra_fused_options* opts, bra::FusedProblem* p) {
  if (!opts) return BRA_OK;
  const int wlen = p->wt ? p->Kp : p->H;
  if (opts->x_pitch != 0) {
    if (opts->x_pitch < p->Kp) return BRA_ERR_INVALID;
    p->xp = opts->x_pitch;
  }
  if (opts->w_pitch != 0) {
    if (opts->w_pitch < wlen) return BRA_ERR_INVALID;
    p->wp = opts->w_pitch;
  }
  return BRA_OK;
}

bool pitched(const bra::FusedProblem& p) {
  return p.xp != p.Kp || p.wp != (p.wt ? p.Kp : p.H);
}

// Byte ranges of every input and output of a validated problem.
void tensor_ranges(const bra::FusedProblem& p, std::vector<Range>* all) {
  const int64_t P = (int64_t)p.ep * p.tp;
  const int64_t El = p.El, Kp = p.Kp, H = p.H, C = p.C, E = El * p.ep;
  const int64_t bes = p.dtype == BRA_FP16 ? 2 : 4;
  const int64_t Hb = p.type == 0 ? H / p.tp : H;
  // pitched operands: El * rows rows `pitch` elements apart, the last one
  // ending at its row length
  const int64_t xrows = El * p.ep * C, wrows = El * (p.wt ? H : Kp);
  const int64_t wlen = p.wt ? Kp : H;
  const int64_t xb = ((xrows - 1) * p.xp + Kp) * 2, wb = ((wrows - 1) * p.wp + wlen) * 2;
  const int64_t bb = El * Hb * bes;
  const int64_t yb = (p.type == 0 ? E * C * (H / p.tp) : E * (C / p.tp) * H) * 2;
  for (int64_t r = 0; r < P; ++r) {
    all->push_back({(uintptr_t)p.x[r], (uintptr_t)p.x[r] + (uintptr_t)xb, false});
    all->push_back({(uintptr_t)p.w[r], (uintptr_t)p.w[r] + (uintptr_t)wb, false});
    if (p.bias) all->push_back({(uintptr_t)p.bias[r], (uintptr_t)p.bias[r] + (uintptr_t)bb, false});
    all->push_back({(uintptr_t)p.y[r], (uintptr_t)p.y[r] + (uintptr_t)yb, true});
  }
}

// The copies the packed variant makes ([CANN] §调用说明 two-phase workspace):
// an operand is copied when its rows lack a 16-byte pitch or a pointer is
// not 16-byte aligned; copies have pitches rounded up to 64 elements (rows
// start on 128-byte L2 lines, so no TMA box row straddles two lines) and
// start 256-byte aligned, x copies of all ranks first, then weight copies.
struct PackPlan {
  bool ok = false;            // the packed variant can take the call
  bool px = false, pw = false;
  int xp = 0, wp = 0;         // pitches of the copies (elements)
  int64_t x_rows = 0, w_rows = 0;
  int64_t xbytes = 0, wbytes = 0;   // one rank's copy, rounded up to 256 bytes
  int64_t total = 0;
};

int64_t round256(int64_t v) { return (v + 255) / 256 * 256; }

PackPlan pack_plan(const bra::FusedProblem& p) {
  PackPlan q;
  const int P = p.ep * p.tp;
  if (P > bra::kMaxRanks) return q;
  auto low = [](const void* a, uintptr_t m) { return (reinterpret_cast<uintptr_t>(a) & m) != 0; };
  const int wlen = p.wt ? p.Kp : p.H;
  q.px = p.Kp % 8 != 0;
  q.pw = wlen % 8 != 0;
  const uintptr_t bias_mask = p.dtype == BRA_BF16 ? 3u : 1u;
  for (int r = 0; r < P; ++r) {
    // element alignment everywhere: the repack reads 16-bit elements, the
    // TMA kernels' element-wise epilogue writes them
    if (low(p.x[r], 1u) || low(p.w[r], 1u) || low(p.y[r], 1u)) return q;
    if (p.bias && low(p.bias[r], bias_mask)) return q;
    if (low(p.x[r], 15u)) q.px = true;
    if (low(p.w[r], 15u)) q.pw = true;
  }
  q.ok = true;
  q.xp = (p.Kp + 63) / 64 * 64;
  q.wp = (wlen + 63) / 64 * 64;
  q.x_rows = (int64_t)p.El * p.ep * p.C;
  q.w_rows = (int64_t)p.El * (p.wt ? p.H : p.Kp);
  q.xbytes = round256(q.x_rows * q.xp * 2);
  q.wbytes = round256(q.w_rows * q.wp * 2);
  q.total = (int64_t)P * ((q.px ? q.xbytes : 0) + (q.pw ? q.wbytes : 0));
  return q;
}

// BRA_FORCE_VARIANT=tc|tc2|tcr|tcu|simt, read at every call.
int forced_variant() {
  const char* v = std::getenv("BRA_FORCE_VARIANT");
  if (!v || !*v) return BRA_VARIANT_AUTO;
  if (!std::strcmp(v, "tc")) return BRA_VARIANT_TC;
  if (!std::strcmp(v, "tc2")) return BRA_VARIANT_TC2;
  if (!std::strcmp(v, "simt")) return BRA_VARIANT_SIMT;
  if (!std::strcmp(v, "tcu")) return BRA_VARIANT_TCU;
  if (!std::strcmp(v, "tcr")) return BRA_VARIANT_TCR;
  if (!std::strcmp(v, "packed")) return BRA_VARIANT_PACKED;
  return BRA_VARIANT_AUTO;
}

// The CTA-pair kernel moves a third less shared-memory traffic per FLOP;
// with few 256 x 256 tiles the one-CTA kernel spreads over more SMs, and
// with at most 128 token rows per group (a weight-streaming, HBM-bound
// problem) the pair's 256-row tile would be half empty.
int tma_kernel_for(const bra::FusedProblem& p) {
  const int64_t rows = (int64_t)p.ep * p.C;
  const int64_t pair_tiles = (int64_t)p.ep * p.El * ((rows + 255) / 256) *
                             (((int64_t)p.H + 255) / 256);
  return pair_tiles >= 64 && rows > 128 ? BRA_VARIANT_TC2 : BRA_VARIANT_TC;
}

// The packed variant for a call that gives `opts`: BRA_VARIANT_PACKED, or a
// negative status (no workspace where one is needed: UNSUPPORTED; one too
// small: INVALID).
int packed_or_status(const bra::FusedProblem& p, const bra_fused_options* opts) {
  const PackPlan q = pack_plan(p);
  if (!q.ok) return -BRA_ERR_UNSUPPORTED;
  if (q.total == 0) return BRA_VARIANT_PACKED;
  if (!opts || !opts->workspace) return -BRA_ERR_UNSUPPORTED;
  return opts->workspace_bytes >= q.total ? BRA_VARIANT_PACKED : -BRA_ERR_INVALID;
}

int choose_variant(const bra::FusedProblem& p, const bra_fused_options* opts) {
  const int f = (opts && opts->variant != BRA_VARIANT_AUTO) ? opts->variant : forced_variant();
  const bool tc_ok = bra::fused_tc_eligible(p);
  const bool tcu_ok = bra::fused_tcu_eligible(p);
  const bool tcr_ok = bra::fused_tcr_eligible(p);
  // Caller-pitched operands: the TMA kernels, or the row-class kernel for
  // other pitches (both address rows only through tensor maps); the
  // load-staged and generic kernels and the repack read dense rows.
  if (pitched(p)) {
    if (f == BRA_VARIANT_TC || f == BRA_VARIANT_TC2) return tc_ok ? f : -BRA_ERR_UNSUPPORTED;
    if (f == BRA_VARIANT_TCR) return tcr_ok ? f : -BRA_ERR_UNSUPPORTED;
    if (f != BRA_VARIANT_AUTO) return -BRA_ERR_UNSUPPORTED;
    return tc_ok ? tma_kernel_for(p) : tcr_ok ? BRA_VARIANT_TCR : -BRA_ERR_UNSUPPORTED;
  }
  if (f == BRA_VARIANT_SIMT) return BRA_VARIANT_SIMT;
  if (f == BRA_VARIANT_TC || f == BRA_VARIANT_TC2) return tc_ok ? f : -BRA_ERR_UNSUPPORTED;
  if (f == BRA_VARIANT_TCU) return tcu_ok ? f : -BRA_ERR_UNSUPPORTED;
  if (f == BRA_VARIANT_TCR) return tcr_ok ? f : -BRA_ERR_UNSUPPORTED;
  if (f == BRA_VARIANT_PACKED) return packed_or_status(p, opts);
  // Rows without a 16-byte pitch: with a workspace, the operands repacked
  // for the TMA kernel; otherwise the CTA-pair kernel fed by row-class TMA
  // maps; when a launch cannot hold the maps of one TP group, the kernel
  // that stages operands with loads; pointers not even element-aligned: the
  // generic kernel.
  if (!tc_ok) {
    if (opts && opts->workspace && pack_plan(p).ok) return packed_or_status(p, opts);
    return tcr_ok ? BRA_VARIANT_TCR : tcu_ok ? BRA_VARIANT_TCU : BRA_VARIANT_SIMT;
  }
  return tma_kernel_for(p);
}

bool log_enabled();

// Repack the operands the plan names into the workspace (after checking
// that it overlaps no input or output), then run the TMA kernel on the
// copies.  Everything is enqueued on `st`.
int run_packed(const bra::FusedProblem& p, const bra_fused_options* opts, cudaStream_t st) {
  const PackPlan q = pack_plan(p);
  if (!q.ok) return BRA_ERR_UNSUPPORTED;
  const int P = p.ep * p.tp;
  std::vector<const void*> xs(p.x, p.x + P), wsrc(p.w, p.w + P);
  if (q.total > 0) {
    std::vector<Range> all;
    tensor_ranges(p, &all);
    const uintptr_t lo = reinterpret_cast<uintptr_t>(opts->workspace);
    const uintptr_t hi = lo + (uintptr_t)q.total;
    for (const Range& a : all)
      if (a.lo < hi && lo < a.hi) return BRA_ERR_INVALID;
    bra::RepackArgs a;
    std::memset(&a, 0, sizeof(a));
    uint8_t* cur = static_cast<uint8_t*>(opts->workspace);
    cudaError_t e = cudaSuccess;
    auto add = [&](const void* src, void* dst, int64_t rows, int len, int pitch) {
      if (e != cudaSuccess) return;
      if (a.njobs == bra::kRepackJobs) {
        e = bra::launch_repack(a, st);
        a.njobs = 0;
        a.total_rows = 0;
        if (e != cudaSuccess) return;
      }
      a.job[a.njobs++] = bra::RepackJob{src, dst, a.total_rows, len, pitch};
      a.total_rows += rows;
    };
    if (q.px)
      for (int r = 0; r < P; ++r) {
        add(p.x[r], cur, q.x_rows, p.Kp, q.xp);
        xs[r] = cur;
        cur += q.xbytes;
      }
    if (q.pw)
      for (int r = 0; r < P; ++r) {
        add(p.w[r], cur, q.w_rows, p.wt ? p.Kp : p.H, q.wp);
        wsrc[r] = cur;
        cur += q.wbytes;
      }
    if (e == cudaSuccess && a.njobs > 0) e = bra::launch_repack(a, st);
    if (e != cudaSuccess) return BRA_ERR_CUDA;
  }
  bra::FusedProblem r = p;
  r.x = xs.data();
  r.w = wsrc.data();
  if (q.px) r.xp = q.xp;
  if (q.pw) r.wp = q.wp;
  if (!bra::fused_tc_eligible(r)) return BRA_ERR_UNSUPPORTED;
  const int v = tma_kernel_for(r);
  if (log_enabled())
    std::fprintf(stderr, "[bra] packed: x %s (pitch %d), weight %s (pitch %d), %lld bytes -> %s\n",
                 q.px ? "copied" : "in place", r.xp, q.pw ? "copied" : "in place", r.wp,
                 (long long)q.total, v == BRA_VARIANT_TC2 ? "tc2" : "tc");
  const cudaError_t e = v == BRA_VARIANT_TC2 ? bra::launch_fused_tc2(r, st)
                                             : bra::launch_fused_tc(r, st);
  if (e == cudaErrorInvalidValue) return BRA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? BRA_OK : BRA_ERR_CUDA;
}

const char* variant_name(int v) {
  return v == BRA_VARIANT_PACKED ? "packed"
         : v == BRA_VARIANT_TC2 ? "tc2"
         : v == BRA_VARIANT_TC  ? "tc"
         : v == BRA_VARIANT_TCR ? "tcr"
         : v == BRA_VARIANT_TCU ? "tcu"
                                : "simt";
}

bool log_enabled() {
  const char* v = std::getenv("BRA_LOG");
  return v && *v && *v != '0';
}

int a2av_common(const void* const input[], const int64_t* send_counts,
                int64_t* send_displs, int64_t* recv_counts,
                int64_t* recv_displs, void* const out[], int64_t P,
                int64_t core_num, int dtype, const int64_t* out_capacity,
                int32_t* status_dev, bool checked, cudaStream_t stream) {
  if (!input || !send_counts || !send_displs || !recv_counts || !recv_displs || !out)
    return BRA_ERR_NULLPTR;
  if (checked && (!out_capacity || !status_dev)) return BRA_ERR_NULLPTR;
  if (P < 1) return BRA_ERR_INVALID;
  if (core_num < 1 || core_num > kInt32Max) return BRA_ERR_INVALID;
  if (dtype != BRA_FP32 && dtype != BRA_INT8) return BRA_ERR_INVALID;
  if (P > bra::kA2avMaxP) return BRA_ERR_UNSUPPORTED;
  // NULL entries are allowed (a rank with nothing to send or receive may
  // have an empty buffer); the kernel rejects a call that would touch one.
  for (int64_t j = 0; j < P; ++j) {
    if (!out[j]) continue;
    for (int64_t i = 0; i < P; ++i)
      if (out[j] == input[i]) return BRA_ERR_INVALID;
    for (int64_t k = 0; k < j; ++k)
      if (out[j] == out[k]) return BRA_ERR_INVALID;
  }
  const int64_t B = cal_all_to_all_v_blocks(P, core_num);
  if (B < 1 || B * P > kInt32Max) return BRA_ERR_INVALID;

  bra::A2avArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int64_t r = 0; r < P; ++r) {
    a.in[r] = input[r];
    a.out[r] = out[r];
    a.cap[r] = checked ? out_capacity[r] : 0;
    if (!input[r]) a.in_null |= uint64_t(1) << r;
    if (!out[r]) a.out_null |= uint64_t(1) << r;
  }
  a.sc = send_counts;
  a.sd = send_displs;
  a.rc = recv_counts;
  a.rd = recv_displs;
  a.status = checked ? status_dev : nullptr;
  a.P = (int)P;
  a.esize = dtype == BRA_FP32 ? 4 : 1;
  a.check_cap = checked ? 1 : 0;
  const int blocks = bra::a2av_launch_blocks(B);
  if (blocks < 1) return BRA_ERR_CUDA;
  if (log_enabled())
    std::fprintf(stderr, "[bra] all_to_all_v P=%lld L=%lld B=%lld blocks=%d\n", (long long)P,
                 (long long)core_num, (long long)B, blocks);
  cudaError_t e = bra::launch_a2av(a, blocks, stream);
  return e == cudaSuccess ? BRA_OK : BRA_ERR_CUDA;
}

int ia2av_common(const void* const input[], const int64_t in_len[],
                 const int64_t* const index[], const int64_t* send_counts,
                 int64_t* send_displs, int64_t* recv_counts, int64_t* recv_displs,
                 void* const out[], int64_t P, int64_t core_num, int dtype,
                 int32_t* status_dev, cudaStream_t stream) {
  if (!input || !in_len || !index || !send_counts || !send_displs || !recv_counts ||
      !recv_displs || !out)
    return BRA_ERR_NULLPTR;
  if (P < 1) return BRA_ERR_INVALID;
  if (core_num < 1 || core_num > kInt32Max) return BRA_ERR_INVALID;
  if (dtype != BRA_FP32 && dtype != BRA_INT8) return BRA_ERR_INVALID;
  if (P > bra::kA2avMaxP) return BRA_ERR_UNSUPPORTED;
  for (int64_t i = 0; i < P; ++i) {
    if (in_len[i] < 0) return BRA_ERR_INVALID;
    if (in_len[i] > 0 && !input[i]) return BRA_ERR_NULLPTR;
  }
  // An output may alias no input, no index array and no other output.
  for (int64_t j = 0; j < P; ++j) {
    if (!out[j]) continue;
    for (int64_t i = 0; i < P; ++i)
      if (out[j] == input[i] || out[j] == static_cast<const void*>(index[i]))
        return BRA_ERR_INVALID;
    for (int64_t k = 0; k < j; ++k)
      if (out[j] == out[k]) return BRA_ERR_INVALID;
  }
  const int64_t B = cal_all_to_all_v_blocks(P, core_num);
  if (B < 1 || B * P > kInt32Max) return BRA_ERR_INVALID;

  bra::IA2avArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int64_t r = 0; r < P; ++r) {
    a.in[r] = input[r];
    a.idx[r] = index[r];
    a.in_len[r] = in_len[r];
    a.out[r] = out[r];
  }
  a.sc = send_counts;
  a.sd = send_displs;
  a.rc = recv_counts;
  a.rd = recv_displs;
  a.status = status_dev;
  a.P = (int)P;
  a.esize = dtype == BRA_FP32 ? 4 : 1;
  const int blocks = bra::ia2av_launch_blocks(core_num);
  if (blocks < 1) return BRA_ERR_CUDA;
  if (log_enabled())
    std::fprintf(stderr, "[bra] indexed_all_to_all_v P=%lld L=%lld blocks=%d\n", (long long)P,
                 (long long)core_num, blocks);
  cudaError_t e = cudaSuccess;
  if (status_dev) e = cudaMemsetAsync(status_dev, 0, sizeof(int32_t), stream);
  if (e == cudaSuccess) e = bra::launch_ia2av(a, blocks, stream);
  return e == cudaSuccess ? BRA_OK : BRA_ERR_CUDA;
}

}  // namespace

extern "C" {

int indexed_all_to_all_v(const void* const input[], const int64_t in_len[],
                         const int64_t* const index[], const int64_t* send_counts,
                         int64_t* send_displs, int64_t* recv_counts, int64_t* recv_displs,
                         void* const out[], int64_t P, int64_t core_num, int dtype,
                         int32_t* status_dev, bra_stream_t stream) {
  return ia2av_common(input, in_len, index, send_counts, send_displs, recv_counts, recv_displs,
                      out, P, core_num, dtype, status_dev, (cudaStream_t)stream);
}

int bmm_rs_a2a_ex(const void* const x[], const void* const weight[],
                  const void* const bias[], int64_t ep, int64_t tp, int64_t E,
                  int64_t C, int64_t M, int64_t H, int64_t yShardType, int dtype,
                  void* const out[], const bra_fused_options* opts, bra_stream_t stream) {
  bra::FusedProblem p;
  int rc = validate_fused(x, weight, bias, ep, tp, E, C, M, H, yShardType, dtype, out, opts, &p);
  if (rc != BRA_OK) return rc;
  const int v = choose_variant(p, opts);
  if (v < 0) return -v;
  if (log_enabled())
    std::fprintf(stderr,
                 "[bra] bmm_rs_a2a ep=%lld tp=%lld E=%lld C=%lld M=%lld H=%lld type=%lld -> %s%s\n",
                 (long long)ep, (long long)tp, (long long)E, (long long)C, (long long)M,
                 (long long)H, (long long)yShardType, variant_name(v),
                 v != BRA_VARIANT_TC2                ? ""
                 : bra::fused_tc2_tile_n(p) == 512 ? (bra::fused_tc2_share(p)
                                                          ? " (256x512 tiles, weight boxes shared)"
                                                          : " (256x512 tiles)")
                 : bra::fused_tc2_share(p)         ? " (256x256 tiles, weight boxes shared)"
                                                   : " (256x256 tiles)");
  if (p.status && cudaMemsetAsync(p.status, 0, sizeof(int32_t), (cudaStream_t)stream) !=
                      cudaSuccess)
    return BRA_ERR_CUDA;
  if (v == BRA_VARIANT_PACKED) return run_packed(p, opts, (cudaStream_t)stream);
  cudaError_t e = v == BRA_VARIANT_TC2   ? bra::launch_fused_tc2(p, (cudaStream_t)stream)
                  : v == BRA_VARIANT_TC  ? bra::launch_fused_tc(p, (cudaStream_t)stream)
                  : v == BRA_VARIANT_TCR ? bra::launch_fused_tcr(p, (cudaStream_t)stream)
                  : v == BRA_VARIANT_TCU ? bra::launch_fused_tcu(p, (cudaStream_t)stream)
                                        : bra::launch_fused_simt(p, (cudaStream_t)stream);
  if (e == cudaErrorInvalidValue && v != BRA_VARIANT_SIMT) return BRA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? BRA_OK : BRA_ERR_CUDA;
}

int bmm_rs_a2a(const void* const x[], const void* const weight[],
               const void* const bias[], int64_t ep, int64_t tp, int64_t E,
               int64_t C, int64_t M, int64_t H, int64_t yShardType, int dtype,
               void* const out[], bra_stream_t stream) {
  return bmm_rs_a2a_ex(x, weight, bias, ep, tp, E, C, M, H, yShardType, dtype, out, nullptr,
                       stream);
}

int bmm_rs_a2a_variant(const void* const x[], const void* const weight[],
                       const void* const bias[], int64_t ep, int64_t tp,
                       int64_t E, int64_t C, int64_t M, int64_t H,
                       int64_t yShardType, int dtype, void* const out[],
                       const bra_fused_options* opts) {
  bra::FusedProblem p;
  int rc = validate_fused(x, weight, bias, ep, tp, E, C, M, H, yShardType, dtype, out, opts, &p);
  if (rc != BRA_OK) return -rc;
  return choose_variant(p, opts);
}

int64_t bmm_rs_a2a_workspace_size(const void* const x[], const void* const weight[],
                                  const void* const bias[], int64_t ep, int64_t tp, int64_t E,
                                  int64_t C, int64_t M, int64_t H, int64_t yShardType,
                                  int dtype, void* const out[], const bra_fused_options* opts) {
  bra_fused_options o;
  std::memset(&o, 0, sizeof(o));
  if (opts) o = *opts;
  o.workspace = nullptr;
  o.workspace_bytes = 0;
  bra::FusedProblem p;
  const int rc = validate_fused(x, weight, bias, ep, tp, E, C, M, H, yShardType, dtype, out, &o,
                                &p);
  if (rc != BRA_OK) return -rc;
  if (bra::fused_tc_eligible(p) || pitched(p)) return 0;
  const PackPlan q = pack_plan(p);
  return q.ok ? q.total : 0;
}

int bmm_rs_a2a_infer_shape(int64_t ep, int64_t tp, int64_t E, int64_t C,
                           int64_t M, int64_t H, int64_t yShardType,
                           int64_t x_shape[3], int64_t w_shape[3],
                           int64_t bias_shape[3], int64_t y_shape[3]) {
  int rc = check_fused_attrs(ep, tp, E, C, M, H, yShardType);
  if (rc != BRA_OK) return rc;
  const int64_t El = E / ep, Kp = M / tp;
  if (x_shape) {
    x_shape[0] = El;
    x_shape[1] = ep * C;
    x_shape[2] = Kp;
  }
  if (w_shape) {
    w_shape[0] = El;
    w_shape[1] = Kp;
    w_shape[2] = H;
  }
  if (bias_shape) {
    bias_shape[0] = El;
    bias_shape[1] = 1;
    bias_shape[2] = yShardType == 0 ? H / tp : H;
  }
  if (y_shape) {
    y_shape[0] = E;
    y_shape[1] = yShardType == 0 ? C : C / tp;
    y_shape[2] = yShardType == 0 ? H / tp : H;
  }
  return BRA_OK;
}

int64_t cal_all_to_all_v_blocks(int64_t P, int64_t L) {
  if (P < 1 || L < 1 || L > kInt32Max) return -1;
  if (L < P) return L;
  return (L / P) * P;
}

int64_t all_to_all_v_launch_blocks(int64_t P, int64_t L) {
  if (P < 1 || L < 1 || L > kInt32Max) return -BRA_ERR_INVALID;
  if (P > bra::kA2avMaxP) return -BRA_ERR_UNSUPPORTED;
  const int64_t B = cal_all_to_all_v_blocks(P, L);
  if (B < 1 || B * P > kInt32Max) return -BRA_ERR_INVALID;
  const int n = bra::a2av_launch_blocks(B);
  return n < 1 ? -BRA_ERR_CUDA : n;
}

int all_to_all_v(const void* const input[], const int64_t* send_counts,
                 int64_t* send_displs, int64_t* recv_counts,
                 int64_t* recv_displs, void* const out[], int64_t P,
                 int64_t core_num, int dtype, bra_stream_t stream) {
  return a2av_common(input, send_counts, send_displs, recv_counts, recv_displs,
                     out, P, core_num, dtype, nullptr, nullptr, false,
                     (cudaStream_t)stream);
}

int all_to_all_v_checked(const void* const input[], const int64_t* send_counts,
                         int64_t* send_displs, int64_t* recv_counts,
                         int64_t* recv_displs, void* const out[], int64_t P,
                         int64_t core_num, int dtype,
                         const int64_t* out_capacity, int32_t* status_dev,
                         bra_stream_t stream) {
  return a2av_common(input, send_counts, send_displs, recv_counts, recv_displs,
                     out, P, core_num, dtype, out_capacity, status_dev, true,
                     (cudaStream_t)stream);
}

const char* bra_status_str(int status) {
  switch (status) {
    case BRA_OK: return "BRA_OK";
    case BRA_ERR_NULLPTR: return "BRA_ERR_NULLPTR";
    case BRA_ERR_INVALID: return "BRA_ERR_INVALID";
    case BRA_ERR_UNSUPPORTED: return "BRA_ERR_UNSUPPORTED";
    case BRA_ERR_CUDA: return "BRA_ERR_CUDA";
    case BRA_ERR_TIMEOUT: return "BRA_ERR_TIMEOUT";
    default: return "BRA_UNKNOWN_STATUS";
  }
}

int bra_l2_flush(void* buf, size_t bytes, bra_stream_t stream) {
  if (!buf) return BRA_ERR_NULLPTR;
  if (reinterpret_cast<uintptr_t>(buf) & 15u) return BRA_ERR_INVALID;
  cudaError_t e = bra::launch_l2_flush(buf, bytes, (cudaStream_t)stream);
  return e == cudaSuccess ? BRA_OK : BRA_ERR_CUDA;
}

int bra_fault_status(int32_t* code, int clear) {
  if (!code) return BRA_ERR_NULLPTR;
  int32_t a = 0, b = 0, c = 0, d = 0, g = 0;
  if (bra::read_fault_word(&a, clear) != cudaSuccess) return BRA_ERR_CUDA;
  if (bra::read_fault_word2(&c, clear) != cudaSuccess) return BRA_ERR_CUDA;
  if (bra::read_fault_word3(&d, clear) != cudaSuccess) return BRA_ERR_CUDA;
  if (bra::read_fault_word4(&g, clear) != cudaSuccess) return BRA_ERR_CUDA;
  if (bra::read_a2av_fault_word(&b, clear) != cudaSuccess) return BRA_ERR_CUDA;
  *code = a ? a : c ? c : d ? d : g ? g : b;
  return BRA_OK;
}

int bra_wait_selftest(int which, int32_t* status_dev, bra_stream_t stream) {
  if (!status_dev) return BRA_ERR_NULLPTR;
  cudaError_t e;
  if (which == BRA_WAIT_A2AV)
    e = bra::launch_a2av_wait_probe(status_dev, (cudaStream_t)stream);
  else if (which == BRA_WAIT_TC)
    e = bra::launch_tc_wait_probe(status_dev, (cudaStream_t)stream);
  else if (which == BRA_WAIT_TC_CLUSTER)
    e = bra::launch_tcr_wait_probe(status_dev, (cudaStream_t)stream);
  else
    return BRA_ERR_INVALID;
  return e == cudaSuccess ? BRA_OK : BRA_ERR_CUDA;
}

int bra_mma_rate_probe(int ctas, int iters, int dtype, int64_t* rec_dev, bra_stream_t stream) {
  if (!rec_dev) return BRA_ERR_NULLPTR;
  if (dtype != BRA_FP16 && dtype != BRA_BF16) return BRA_ERR_INVALID;
  if (iters < 1 || iters > (1 << 22)) return BRA_ERR_INVALID;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return BRA_ERR_CUDA;
  if (ctas < 1 || ctas > sms) return BRA_ERR_INVALID;
  const cudaError_t e =
      bra::launch_mma_probe(ctas, iters, dtype == BRA_BF16, rec_dev, (cudaStream_t)stream);
  return e == cudaSuccess ? BRA_OK : BRA_ERR_CUDA;
}

int bra_gather_rate_probe(const void* buf, int64_t bytes, int ctas, int iters, int64_t* rec_dev,
                          bra_stream_t stream) {
  if (!buf || !rec_dev) return BRA_ERR_NULLPTR;
  if (bytes < 4096 || bytes > (int64_t(1) << 40) || (bytes & (bytes - 1)) != 0)
    return BRA_ERR_INVALID;
  if (iters < 1 || iters > (1 << 20)) return BRA_ERR_INVALID;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return BRA_ERR_CUDA;
  if (ctas < 1 || ctas > sms) return BRA_ERR_INVALID;
  const cudaError_t e =
      bra::launch_gather_probe(buf, bytes, ctas, iters, rec_dev, (cudaStream_t)stream);
  return e == cudaSuccess ? BRA_OK : BRA_ERR_CUDA;
}

const char* bra_version(void) { return "0.1.0"; }

}  // extern "C"
