// Internal declarations shared by the host entry points and the kernels of
// libbmmrsa2a.so.  Not installed; the public ABI is include/bmm_rs_a2a.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bmm_rs_a2a.h"

namespace bra {

// all_to_all_v keeps the whole P x P count matrix of int64 in shared memory.
constexpr int kA2avMaxP = 64;

// Fused kernels: one launch covers the TP groups of up to kChunkRanks source
// ranks (their x / weight / bias), and may write to any of kMaxRanks outputs.
constexpr int kChunkRanks = 64;
constexpr int kMaxRanks = 32 * 32;

struct A2avArgs {
  const void* in[kA2avMaxP];
  void* out[kA2avMaxP];
  int64_t cap[kA2avMaxP];   // receive capacity per rank (elements)
  const int64_t* sc;        // send_counts [P][P]
  int64_t* sd;              // send_displs [P][P]
  int64_t* rc;              // recv_counts [P][P]
  int64_t* rd;              // recv_displs [P][P]
  int32_t* status;          // optional device status word
  uint64_t in_null;         // bit r: in[r] is NULL
  uint64_t out_null;        // bit r: out[r] is NULL
  int P;
  int esize;                // element size in bytes (4 or 1)
  int check_cap;            // compare received totals against cap[]
  int stages;               // ring slots per warp (set by launch_a2av)
  uint32_t chunk;           // bytes per chunk (set by launch_a2av)
};

// Blocks the exchange launches for an admitted block count B on the current
// device: B, at most the SM count (one block per SM); -1 if the device
// cannot be queried.
int a2av_launch_blocks(int64_t B);
// Launch the exchange on `blocks` blocks.
cudaError_t launch_a2av(const A2avArgs& a, int blocks, cudaStream_t st);

// Indexed exchange: rank i's send list is input[i] gathered through idx[i].
struct IA2avArgs {
  const void* in[kA2avMaxP];
  const int64_t* idx[kA2avMaxP];
  int64_t in_len[kA2avMaxP];  // elements of in[i]; index values must lie below
  void* out[kA2avMaxP];
  const int64_t* sc;          // send_counts [P][P]
  int64_t* sd;                // send_displs [P][P]
  int64_t* rc;                // recv_counts [P][P]
  int64_t* rd;                // recv_displs [P][P]
  int32_t* status;            // optional device status word
  int P;
  int esize;                  // element size in bytes (4 or 1)
};
// Blocks the indexed exchange launches for core_num L: L, at most the SM
// count (one block per SM); -1 if the device cannot be queried.
int ia2av_launch_blocks(int64_t L);
cudaError_t launch_ia2av(const IA2avArgs& a, int blocks, cudaStream_t st);

// Problem description shared by the fused kernels.
struct FusedProblem {
  const void* const* x;      // [P]
  const void* const* w;      // [P]
  const void* const* bias;   // [P] or nullptr
  void* const* y;            // [P]
  int ep, tp, El, C, Kp, H;
  int type;                  // yShardType
  int dtype;                 // BRA_FP16 | BRA_BF16
  int wt;                    // weight stored transposed: (El, H, Kp)
  // Row pitches in elements: x rows (Kp long) and weight rows (H long, or Kp
  // when transposed).  Equal to the row lengths for the caller's dense
  // tensors; larger for repacked copies, whose rows start 16-byte aligned.
  // Only the TMA kernels (fused_tc*) accept pitches other than the lengths.
  int xp, wp;
  int32_t* status;           // per-call timeout word (optional)
};

cudaError_t launch_fused_simt(const FusedProblem& f, cudaStream_t st);
// Both return cudaErrorInvalidValue if a TMA descriptor cannot be encoded.
cudaError_t launch_fused_tc(const FusedProblem& f, cudaStream_t st);    // one CTA per tile
cudaError_t launch_fused_tc2(const FusedProblem& f, cudaStream_t st);   // CTA pair per tile
// Width of that kernel's pair tiles for this problem: 256 or 512.
int fused_tc2_tile_n(const FusedProblem& f);
// Whether that kernel runs two pairs per cluster sharing each weight box.
int fused_tc2_share(const FusedProblem& f);
// Shape / alignment predicate of the tensor-core variant.
bool fused_tc_eligible(const FusedProblem& f);
// Tensor-core variant for rows of any alignment (operands staged by loads).
cudaError_t launch_fused_tcu(const FusedProblem& f, cudaStream_t st);
bool fused_tcu_eligible(const FusedProblem& f);
// CTA-pair tensor-core variant for rows without a 16-byte pitch, fed by TMA
// through row-class maps (cudaErrorInvalidValue if a map cannot be encoded).
cudaError_t launch_fused_tcr(const FusedProblem& f, cudaStream_t st);
bool fused_tcr_eligible(const FusedProblem& f);

cudaError_t launch_l2_flush(void* buf, size_t bytes, cudaStream_t st);
// Tensor-core rate probe: `ctas` CTAs, one per SM, each iters x 4 MMAs.
cudaError_t launch_mma_probe(int ctas, int iters, bool bf16, int64_t* rec, cudaStream_t st);
// Gather-rate probe: `ctas` CTAs, one per SM, each 1024 threads x iters x 8
// random one-byte loads from buf (bytes a power of two).
cudaError_t launch_gather_probe(const void* buf, int64_t bytes, int ctas, int iters, int64_t* rec,
                                cudaStream_t st);

// Row repacking: copies rows of 16-bit elements that start at any even byte
// address to rows that start 16-byte aligned, `pitch` elements apart.
struct RepackJob {
  const void* src;   // rows of `len` elements, back to back (2-byte aligned)
  void* dst;         // 16-byte aligned; row k starts at dst + k * pitch * 2
  int64_t row0;      // index of this job's first row among all rows of the launch
  int32_t len;       // elements per row
  int32_t pitch;     // destination row pitch in elements (a multiple of 8, > len if len is odd)
};
constexpr int kRepackJobs = 256;
struct RepackArgs {
  RepackJob job[kRepackJobs];   // ordered by row0; job[0].row0 == 0
  int64_t total_rows;
  int njobs;
};
cudaError_t launch_repack(const RepackArgs& a, cudaStream_t st);
cudaError_t read_fault_word(int32_t* code, int clear);        // tensor-core kernel
cudaError_t read_fault_word2(int32_t* code, int clear);       // CTA-pair tensor-core kernel
cudaError_t read_fault_word3(int32_t* code, int clear);       // load-staged unaligned kernel
cudaError_t read_fault_word4(int32_t* code, int clear);       // row-class TMA unaligned kernel
cudaError_t read_a2av_fault_word(int32_t* code, int clear);   // all_to_all_v kernel
// One bounded wait that nothing completes, with each family's wait helper.
cudaError_t launch_a2av_wait_probe(int32_t* status, cudaStream_t st);
cudaError_t launch_tc_wait_probe(int32_t* status, cudaStream_t st);
cudaError_t launch_tcr_wait_probe(int32_t* status, cudaStream_t st);   // cluster-scope wait

}  // namespace bra
