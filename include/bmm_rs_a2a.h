/*
 * bmm_rs_a2a.h -- C ABI of libbmmrsa2a.so: the MoE expert-parallel x
 * tensor-parallel dataflow BatchMatMul -> TP ReduceScatter -> bias Add -> EP
 * AllToAll, the variable-count all_to_all_v exchange and its indexed form,
 * with all ep*tp ranks resident on one GPU as virtual ranks (one buffer
 * partition per rank).
 *
 * Pages cited (by title and section):
 *   [CANN] "CANN ops-transformer 通算融合算子实战 BatchMatMulReduceScatterAllToAll
 *          原理、shape 约束与 aclnn 两段式调用"
 *   [PTO]  "LowerL2TensorCollectives Pass" (PyPTO)
 *   [VCCL] "vccl alltoallv dev log"
 *
 * Conventions shared by every entry point
 *   - Virtual rank r = s*tp + t: s is the rank's EP index, t its TP index
 *     ([CANN] §完整调用示例 step 2: EP groups {t, t+tp, ...}, TP groups
 *     {s*tp .. s*tp+tp-1}).
 *   - Every tensor is dense, row-major (C order), with no padding.
 *   - Device pointers are CUDA device (or managed) addresses on the current
 *     device; the caller owns every buffer and the stream.  The library
 *     allocates no device memory on any call path.
 *   - Work is enqueued on `stream` (NULL = legacy default stream) and runs
 *     asynchronously.  The return value reports argument validation and the
 *     launch itself, not completion; on any error nothing is launched unless
 *     the code is BRA_ERR_CUDA from the launch.
 *   - Calls keep no state from one call to the next, so calls whose outputs
 *     are disjoint may run concurrently on different streams.  Two things
 *     are shared: the watchdog words that bra_fault_status reads (one set
 *     per device, written by any call whose bounded wait gave up, on any
 *     stream; for a word of one call's own, use the status of
 *     all_to_all_v_checked, indexed_all_to_all_v or bra_fused_options), and
 *     the scratch array of bmm_rs_a2a_noalloc.
 *   - Functions are thread-safe.
 */
#ifndef BMM_RS_A2A_H
#define BMM_RS_A2A_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(BRA_BUILD) && defined(__GNUC__)
#define BRA_API __attribute__((visibility("default")))
#else
#define BRA_API
#endif

struct CUstream_st;
typedef struct CUstream_st* bra_stream_t;   /* same type as cudaStream_t */

/* Status codes.  NULLPTR and INVALID keep the values of the aclnn codes
 * ACLNN_ERR_PARAM_NULLPTR / ACLNN_ERR_PARAM_INVALID ([CANN] §调用说明). */
typedef enum {
  BRA_OK = 0,
  BRA_ERR_NULLPTR = 161001,     /* a required pointer is NULL                 */
  BRA_ERR_INVALID = 161002,     /* dtype, attribute, shape or aliasing rule   */
  BRA_ERR_UNSUPPORTED = 161003, /* valid per the pages, beyond the library limits */
  BRA_ERR_CUDA = 161100,        /* a CUDA call failed (launch or query)       */
  BRA_ERR_TIMEOUT = 161101      /* a kernel gave up a bounded wait            */
} bra_status;

typedef enum { BRA_FP16 = 0, BRA_BF16 = 1, BRA_FP32 = 2, BRA_INT8 = 3 } bra_dtype;

/* Kernel variants of bmm_rs_a2a (see bmm_rs_a2a_variant). */
typedef enum {
  BRA_VARIANT_AUTO = 0,
  BRA_VARIANT_TC = 1,    /* tcgen05 / TMEM / TMA kernel, one CTA per tile  */
  BRA_VARIANT_SIMT = 2,  /* generic kernel: any alignment, any size        */
  BRA_VARIANT_TC2 = 3,   /* tcgen05 kernel, a CTA pair per 256x256 or 256x512 tile */
  BRA_VARIANT_TCU = 4,   /* tcgen05 kernel for rows of any alignment:
                            operands staged by loads, not TMA             */
  BRA_VARIANT_TCR = 5,   /* tcgen05 CTA-pair kernel for rows of any
                            alignment: row-class TMA maps, rows shifted
                            into place in shared memory                   */
  BRA_VARIANT_PACKED = 6 /* operands without a 16-byte row pitch copied
                            into the caller's workspace with one, then the
                            TMA kernel (TC or TC2 by the same rule)       */
} bra_variant;

/* ------------------------------------------------------------------------ */
/* Fused BatchMatMul -> ReduceScatter -> Add -> AllToAll                     */
/* ------------------------------------------------------------------------ */

/*
 * bmm_rs_a2a -- [CANN] §功能说明与计算流程:
 *     temp1 = BatchMatMul(x, weight); temp2 = ReduceScatter(temp1) over the
 *     TP group (sum); temp3 = Add(temp2, bias); y = AllToAll(temp3) over the
 *     EP group,
 * computed for all P = ep*tp virtual ranks in one launch, writing straight
 * into every rank's final y; no intermediate reaches memory.
 *
 * Arguments (El = E/ep, Kp = M/tp, Hp = H/tp, Cp = C/tp):
 *   x[P]      device, x[r] of shape (El, ep*C, Kp), dtype `dtype`
 *             (yShardType 1 writes dim 1 as ep*tp*C/tp: the same length).
 *   weight[P] device, weight[r] of shape (El, Kp, H), dtype `dtype`.
 *   bias[P]   NULL, or an array whose entries are all NULL (no bias), or all
 *             non-NULL: bias[r] of shape (El, 1, Hp) / (El, Hp) for
 *             yShardType 0 and (El, 1, H) / (El, H) for yShardType 1 (2-D and
 *             3-D forms share one memory layout); fp16 when dtype is FP16,
 *             fp32 when dtype is BF16 ([CANN] §参数说明).
 *   ep, tp    EP and TP group sizes, each in {1, 2, 4, 8, 16, 32}; the pages
 *             allow {2..32}, 1 is accepted as the degenerate case.
 *   E, C, M, H  as in [CANN] §约束说明.
 *   yShardType 0: reduce-scatter along H; 1: along C.
 *   dtype     BRA_FP16 or BRA_BF16 (x, weight and y).
 *   out[P]    device, y[r] of shape (E, C, Hp) for yShardType 0 and
 *             (E, Cp, H) for yShardType 1, dtype `dtype`.
 *   stream    CUDA stream.
 * Semantics (receiver d = j*tp + t, stacked block i = s*El + e):
 *   Z_{s,e} = sum_{t'=0..tp-1} x[s*tp+t'][e] @ weight[s*tp+t'][e], summed in
 *   fp32 in t' order, shape (ep*C, H);
 *   yShardType 0: y[d][i, c, h]  = Z_{s,e}[j*C + c, t*Hp + h] + bias[s*tp+t][e, h]
 *   yShardType 1: y[d][i, c, h]  = Z_{s,e}[j*C + t*Cp + c, h] + bias[s*tp+t][e, h]
 *   (the bias add is fp32, then one round-to-nearest-even to dtype).
 * Errors (checked in the order of [CANN] §op_api 层 CheckParams; nothing is
 * launched on error):
 *   BRA_ERR_NULLPTR  x, weight or out (the arrays or any entry) is NULL.
 *   BRA_ERR_INVALID  dtype not FP16/BF16; ep or tp not in the set above;
 *                    yShardType not 0/1; E outside [2,512] or not a multiple
 *                    of ep; E/ep outside [1,32]; H outside [1,65535]; M not
 *                    a multiple of tp or M/tp outside [1,65535]; C <= 0;
 *                    yShardType 0 with H % tp != 0; yShardType 1 with
 *                    C % tp != 0 ([CANN] §数据关系与取值范围说明); some but not
 *                    all bias entries NULL; an output range overlapping any
 *                    input range or another output range.
 *   BRA_ERR_UNSUPPORTED  ep*C >= 2^31.
 *   BRA_ERR_CUDA     the launch failed (cudaGetLastError).
 * Variant: when the operands' rows and pointers are 16-byte aligned (Kp % 8
 * == 0, the weight's row length H -- Kp when transposed -- % 8 == 0, x and
 * weight 16-byte aligned) a TMA-fed tensor-core kernel runs: the CTA-pair
 * kernel when the problem has at least 64 output tiles of 256 x 256 and
 * more than 128 token rows (ep*C) per expert group, else the one-CTA
 * kernel.  The CTA pair computes 256 x 512 tiles when the K loop is long
 * (tp * Kp >= 8192), H >= 1024 and there are at least 38 such tiles, else
 * 256 x 256 tiles (the environment variable BRA_TC2_WIDE=1 or 0, read at
 * every call, forces one; BRA_TC2_SHARE=1 runs it as clusters of two pairs
 * that share each weight box by TMA multicast, an option measured no faster
 * and off by default).  Its epilogue stores 16-byte vectors from 16-byte rows when the
 * outputs and bias are 16-byte aligned (and Hp % 8 == 0 for yShardType 0),
 * else it stages each row segment at its destination's 16-byte phase and
 * stores the aligned part as vectors (outputs and bias element-aligned).
 * Other shapes
 * with element-aligned pointers run, given a workspace (bmm_rs_a2a_ex), the
 * packed variant: those operands repacked, then the same TMA kernel.
 * Without a workspace they run the CTA-pair tensor-core kernel fed by
 * row-class TMA maps (one map per
 * class of rows that start at the same offset past a 16-byte boundary, the
 * rows shifted into place in shared memory); when the maps of one TP group
 * do not fit a launch ((n_x + n_w) * tp > 176, n = 1, 2, 4 or 8 classes per
 * operand) the tensor-core kernel that stages operands with loads runs
 * instead.  Pointers that are not even element-aligned run the generic
 * kernel.  Each launches once per 64 source ranks (the row-class kernel once
 * per 176 / (n_x + n_w) ranks).
 * The environment variable BRA_FORCE_VARIANT=tc|tc2|tcr|tcu|simt|packed
 * overrides the choice (tc, tc2, tcr or tcu on an ineligible shape, or
 * packed without a large enough workspace, returns BRA_ERR_UNSUPPORTED).
 */
BRA_API int bmm_rs_a2a(const void* const x[], const void* const weight[],
               const void* const bias[], int64_t ep, int64_t tp, int64_t E,
               int64_t C, int64_t M, int64_t H, int64_t yShardType, int dtype,
               void* const out[], bra_stream_t stream);

/* Options of bmm_rs_a2a_ex.  Zero-initialise; unused fields must stay 0. */
typedef struct {
  /* Non-zero: weight[r] is stored transposed, as (El, H, Kp) row-major (the
   * layout of a view of the (El, Kp, H) weight with its last two dims
   * swapped, the transpose_weight attribute of [CANN] §参数说明 / §op_api 层
   * TransTensor).  The values are the same; only the storage differs. */
  int32_t transpose_weight;
  /* BRA_VARIANT_AUTO (0) or a bra_variant to force; takes precedence over
   * the BRA_FORCE_VARIANT environment variable. */
  int32_t variant;
  /* Row pitches, in elements, of x[r] (rows of Kp) and weight[r] (rows of
   * H, or of Kp when transposed); 0 = dense (pitch = row length).  A pitch
   * must be at least the row length; the tensor is then El * rows rows
   * that many elements apart (the layout of a (El, rows, pitch) buffer
   * viewed as (El, rows, length)), and the elements between a row's end and
   * the next row are never read.  Pitched operands run with no copy: on the
   * TMA kernels when TMA-ready (pitch a multiple of 8 elements, pointers
   * 16-byte aligned), else on the row-class kernel (element-aligned
   * pointers, its map limit); otherwise the call returns
   * BRA_ERR_UNSUPPORTED (the load-staged and generic kernels and the packed
   * variant take dense rows only). */
  int32_t x_pitch;
  int32_t w_pitch;
  /* Device memory the call may use as scratch, in the manner of the second
   * call of the two-phase aclnn interface ([CANN] §调用说明: the workspace
   * and its size).  NULL with workspace_bytes 0: no workspace.  Only
   * BRA_VARIANT_PACKED uses it (see bmm_rs_a2a_workspace_size); it must be
   * 256-byte aligned, hold at least that many bytes, and overlap no input or
   * output.  Its contents are scratch: overwritten, never read before being
   * written.  The caller owns it; it must stay allocated until the call's
   * work on `stream` completes. */
  void* workspace;
  int64_t workspace_bytes;
  /* Optional device int32 of this call alone (NULL: none).  Set to BRA_OK on
   * `stream` before the call's kernels; a kernel whose bounded wait gives up
   * then writes BRA_ERR_TIMEOUT to it (its output is then incomplete).
   * Unlike the per-device words bra_fault_status reads, which every call on
   * the device shares, a timeout in another call never reaches it. */
  int32_t* status;
} bra_fused_options;

/*
 * bmm_rs_a2a_ex -- bmm_rs_a2a with options (NULL opts = all defaults, same
 * as bmm_rs_a2a).  Errors as bmm_rs_a2a, plus BRA_ERR_INVALID for an
 * unknown variant, a negative pitch or one below its row length, a
 * workspace that is not
 * 256-byte aligned, a negative workspace_bytes or a non-zero one with a NULL
 * workspace (always checked), a workspace smaller than
 * bmm_rs_a2a_workspace_size or overlapping an input or output (checked when
 * the packed variant would use it), and BRA_ERR_UNSUPPORTED when a forced
 * tensor-core variant cannot take the shape or alignment, or the packed
 * variant is forced without a workspace where one is needed.
 * With a workspace of at least bmm_rs_a2a_workspace_size bytes, AUTO takes
 * BRA_VARIANT_PACKED for every shape whose x or weight rows lack a 16-byte
 * pitch (and whose pointers are element-aligned): the repack kernel copies
 * those operands' rows into the workspace at a pitch of a multiple of 64
 * elements, then the TMA kernel reads the copies (rows past the logical
 * length read as zeros, so the copies need no zero padding).
 */
BRA_API int bmm_rs_a2a_ex(const void* const x[], const void* const weight[],
                          const void* const bias[], int64_t ep, int64_t tp, int64_t E,
                          int64_t C, int64_t M, int64_t H, int64_t yShardType, int dtype,
                          void* const out[], const bra_fused_options* opts,
                          bra_stream_t stream);

/*
 * bmm_rs_a2a_infer_shape -- per-rank shapes from the attributes ([CANN]
 * §约束说明 and the infershape of §op_api 层): yShardType 0 gives
 * y (E, C, H/tp), 1 gives y (E, C/tp, H).  Each output array receives three
 * int64 values (bias in its 3-D form); any output pointer may be NULL.
 * Pure host function.  Returns BRA_OK or BRA_ERR_INVALID (same range rules
 * as bmm_rs_a2a).
 */
BRA_API int bmm_rs_a2a_infer_shape(int64_t ep, int64_t tp, int64_t E, int64_t C,
                           int64_t M, int64_t H, int64_t yShardType,
                           int64_t x_shape[3], int64_t w_shape[3],
                           int64_t bias_shape[3], int64_t y_shape[3]);

/*
 * bmm_rs_a2a_workspace_size -- bytes of workspace the packed variant needs
 * for these arguments (the first call of the two-phase aclnn interface,
 * [CANN] §调用说明, without the executor): for every rank, a copy of x[r]
 * when M/tp % 8 != 0 or x[r] is not 16-byte aligned, and of weight[r] when
 * its row length (H, or M/tp when transposed) % 8 != 0 or weight[r] is not
 * 16-byte aligned, each with rows rounded up to a multiple of 64 elements
 * (128 bytes) and each copy starting 256-byte aligned (x copies of all ranks
 * first, then weight copies).  0 when no operand needs a copy (the
 * TMA kernels read the caller's tensors) or when the packed variant cannot
 * take the call (a pointer not element-aligned, more than 1024 ranks).  The
 * workspace fields of opts are ignored.  Returns the size, or a negative
 * bra_status when bmm_rs_a2a_ex would reject the arguments.  Pure host.
 */
BRA_API int64_t bmm_rs_a2a_workspace_size(const void* const x[], const void* const weight[],
                                          const void* const bias[], int64_t ep, int64_t tp,
                                          int64_t E, int64_t C, int64_t M, int64_t H,
                                          int64_t yShardType, int dtype, void* const out[],
                                          const bra_fused_options* opts);

/*
 * bmm_rs_a2a_noalloc -- bmm_rs_a2a_ex forced to BRA_VARIANT_PACKED, with
 * scratch memory the library holds itself instead of a caller workspace.
 * The pages have no counterpart: the CANN op always takes its workspace
 * from the caller.
 *
 * Who it is for: callers that cannot allocate device memory for a
 * workspace -- a plugin inside a host program that owns all device memory
 * and hands its plugins only their inputs and outputs, or a path that must
 * not call cudaMalloc because cudaMalloc may synchronise the device.  The
 * call allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine runs on its path.  The caller still passes every input and output.
 *
 * Scratch: one file-scope device array of BRA_NOALLOC_SCRATCH_BYTES
 * (32 MiB), loaded with the library on every device that uses it and held
 * there until the process exits.  The first call on a device, with that
 * device current, looks up the array's address (cudaGetSymbolAddress) and
 * keeps it; make that first call before any stream capture.  Every call on
 * a device shares the array, and the array keeps the last call's contents
 * (nothing in it has to start at zero: the repack writes every byte the
 * TMA kernel reads).  Calls whose work overlaps on the GPU (different
 * streams, no ordering between them) race on the array and give wrong
 * results: order them on one stream or with events.
 *
 * Arguments: as bmm_rs_a2a; transpose_weight non-zero means weight[r] is
 * stored as (El, H, Kp) (the bra_fused_options field of that name).
 * Operands must be dense (no pitch).  Operands whose rows have a 16-byte
 * pitch and 16-byte aligned pointers are not copied and use no scratch.
 * Errors: as bmm_rs_a2a_ex with BRA_VARIANT_PACKED forced; plus
 * BRA_ERR_UNSUPPORTED when the copies need more than
 * BRA_NOALLOC_SCRATCH_BYTES (bmm_rs_a2a_workspace_size gives the need) or
 * the current device's ordinal is 64 or more, and BRA_ERR_CUDA when the
 * array's address cannot be obtained.
 */
#define BRA_NOALLOC_SCRATCH_BYTES (32u << 20)
BRA_API int bmm_rs_a2a_noalloc(const void* const x[], const void* const weight[],
                               const void* const bias[], int64_t ep, int64_t tp, int64_t E,
                               int64_t C, int64_t M, int64_t H, int64_t yShardType, int dtype,
                               void* const out[], int transpose_weight, bra_stream_t stream);

/*
 * bmm_rs_a2a_variant -- which kernel bmm_rs_a2a_ex would launch for these
 * arguments and options (BRA_VARIANT_TC, BRA_VARIANT_TC2, BRA_VARIANT_TCR,
 * BRA_VARIANT_TCU, BRA_VARIANT_SIMT or BRA_VARIANT_PACKED), honouring
 * BRA_FORCE_VARIANT.  Pointers are only
 * inspected for alignment.  Returns the variant, or a negative bra_status
 * (e.g. -BRA_ERR_INVALID) when the call would be rejected.  Pure host.
 */
BRA_API int bmm_rs_a2a_variant(const void* const x[], const void* const weight[],
                       const void* const bias[], int64_t ep, int64_t tp,
                       int64_t E, int64_t C, int64_t M, int64_t H,
                       int64_t yShardType, int dtype, void* const out[],
                       const bra_fused_options* opts);

/* ------------------------------------------------------------------------ */
/* all_to_all_v                                                              */
/* ------------------------------------------------------------------------ */

/*
 * cal_all_to_all_v_blocks -- admitted block count B for P ranks and a
 * requested core_num L ([PTO] §启动宽度): L when L < P, otherwise the
 * largest multiple of P not above L (L=10, P=8 gives 8).  Returns -1 when
 * P < 1 or L is outside [1, INT32_MAX] ([PTO] §约束与诊断).  Pure host.
 */
BRA_API int64_t cal_all_to_all_v_blocks(int64_t P, int64_t L);

/*
 * all_to_all_v_launch_blocks -- thread blocks all_to_all_v and
 * all_to_all_v_checked launch on the current device for P ranks and
 * core_num L: B = cal_all_to_all_v_blocks(P, L), at most the device's SM
 * count.  Each block takes a whole SM (its shared memory leaves room for no
 * other block), so the exchange occupies that many SMs and no more; B above
 * the SM count is clamped because blocks beyond it could not all be resident
 * at once, which [PTO] §启动宽度 requires of the admitted blocks.
 * Returns the count, -BRA_ERR_INVALID for arguments all_to_all_v rejects
 * (P outside [1, 64] gives -BRA_ERR_UNSUPPORTED above 64), or -BRA_ERR_CUDA
 * when the device cannot be queried.  Host function; queries the device.
 */
BRA_API int64_t all_to_all_v_launch_blocks(int64_t P, int64_t L);

/*
 * all_to_all_v -- variable-count exchange among P virtual ranks ([PTO] §行为
 * and §ABI; addressing as in [VCCL] §5 ref): rank i sends send_counts[i][j]
 * elements to rank j, for every pair including i == j:
 *   send_displs[i][j] = sum_{k<j} send_counts[i][k]
 *   recv_counts[j][i] = send_counts[i][j]
 *   recv_displs[j][i] = sum_{k<i} send_counts[k][j]
 *   out[j][recv_displs[j][i] + n] = input[i][send_displs[i][j] + n],
 *       0 <= n < send_counts[i][j]
 * so out[j] holds what rank j received ordered by source rank; its elements
 * past the received total are not written.
 *
 * Arguments:
 *   input[P]     device; input[i] holds at least sum_j send_counts[i][j]
 *                elements of `dtype` (may be NULL when that sum is 0).
 *   send_counts  device, int64 [P][P] row-major (read only).
 *   send_displs, recv_counts, recv_displs
 *                device, int64 [P][P] row-major, written by the kernel.
 *   out[P]       device; out[j] must hold sum_i send_counts[i][j] elements
 *                (the caller's obligation here; see all_to_all_v_checked);
 *                may be NULL when that sum is 0.
 *   P            number of ranks, 1 <= P <= 64.
 *   core_num     requested block count L, in [1, INT32_MAX].  The call
 *                launches B = cal_all_to_all_v_blocks(P, L) thread blocks,
 *                one per SM, at most the SM count
 *                (all_to_all_v_launch_blocks): the exchange occupies B SMs
 *                and leaves the others to concurrent work.  The blocks split
 *                the concatenated send buffers of ranks 0..P-1 into equal
 *                element ranges; results do not depend on B.
 *   dtype        BRA_FP32 or BRA_INT8 ([PTO] §约束与诊断 allowlist).
 * Errors (nothing launched):
 *   BRA_ERR_NULLPTR  input, out, send_counts or a bookkeeping array is NULL.
 *   BRA_ERR_INVALID  P < 1; core_num outside [1, INT32_MAX]; dtype not
 *                    FP32/INT8; an out[j] equal to any input[i] or to another
 *                    out[k] ([PTO] §当前限制: input != target, windows
 *                    pairwise distinct); B*P > INT32_MAX.
 *   BRA_ERR_UNSUPPORTED  P > 64.
 *   BRA_ERR_CUDA     the launch failed.
 * Device-side data check: if any send count is negative, or a NULL
 * input[i] / out[j] would be read / written, the kernel writes nothing at all
 * (no output, no bookkeeping).
 */
BRA_API int all_to_all_v(const void* const input[], const int64_t* send_counts,
                 int64_t* send_displs, int64_t* recv_counts,
                 int64_t* recv_displs, void* const out[], int64_t P,
                 int64_t core_num, int dtype, bra_stream_t stream);

/*
 * all_to_all_v_checked -- all_to_all_v plus device-side checks whose result
 * is written to *status_dev (device int32): BRA_OK, or BRA_ERR_INVALID when a
 * send count is negative, a NULL buffer would be touched, or some rank j
 * would receive more than out_capacity[j] elements; in the error case nothing
 * else is written.
 * out_capacity: host array of P element counts (copied at the call).
 * status_dev: device pointer, required (BRA_ERR_NULLPTR if NULL).
 * The "0 / 1 / capacity / over-capacity / negative" count matrices of
 * [PTO] §测试 map onto this entry point.
 */
BRA_API int all_to_all_v_checked(const void* const input[], const int64_t* send_counts,
                         int64_t* send_displs, int64_t* recv_counts,
                         int64_t* recv_displs, void* const out[], int64_t P,
                         int64_t core_num, int dtype,
                         const int64_t* out_capacity, int32_t* status_dev,
                         bra_stream_t stream);

/*
 * indexed_all_to_all_v -- the URMA indexed exchange ([PTO] §A5 URMA
 * 索引交换).  The page names the operands and says the cores share the local
 * data movement before the remote transfers, but does not define `index`;
 * the reading implemented: rank i's send list is its input gathered through
 * its index, and the send lists are exchanged as in all_to_all_v:
 *   n_i = sum_j send_counts[i][j]
 *   send_i[k] = input[i][index[i][k]],                        0 <= k < n_i
 *   out[j][recv_displs[j][i] + m] = send_i[send_displs[i][j] + m],
 *       0 <= m < send_counts[i][j]
 * with send_displs, recv_counts, recv_displs as in all_to_all_v (written by
 * the kernel).  Elements of out[j] past its received total are not written.
 *
 * Arguments:
 *   input[P]     device; input[i] holds in_len[i] elements of `dtype` (may be
 *                NULL when in_len[i] is 0).
 *   in_len[P]    host; element counts of the inputs (copied at the call).
 *   index[P]     device int64; index[i] holds at least n_i entries (may be
 *                NULL when n_i is 0).
 *   send_counts, send_displs, recv_counts, recv_displs, out, P, dtype
 *                as for all_to_all_v.
 *   core_num     L, in [1, INT32_MAX]: the exact number of blocks the call
 *                launches ([PTO] §A5 URMA 索引交换: L is the exact core
 *                count, not folded by cal_all_to_all_v_blocks), one per SM,
 *                at most the SM count.  The blocks split the send lists of
 *                ranks 0..P-1, taken one after another, into equal position
 *                ranges; results do not depend on L.
 *   status_dev   optional device int32: set to BRA_OK on the stream before
 *                the kernel, then to BRA_ERR_INVALID if the call was rejected
 *                on the device or an index value was out of range.
 * Errors (nothing launched):
 *   BRA_ERR_NULLPTR  input, in_len, index, out, send_counts or a bookkeeping
 *                    array is NULL; input[i] NULL with in_len[i] > 0.
 *   BRA_ERR_INVALID  P < 1; core_num outside [1, INT32_MAX]; dtype not
 *                    FP32/INT8; in_len[i] < 0; an out[j] equal to an input,
 *                    an index array or another output; B*P > INT32_MAX.
 *   BRA_ERR_UNSUPPORTED  P > 64.
 *   BRA_ERR_CUDA     the launch failed.
 * Device-side data checks: a negative send count, or a NULL index[i] /
 * out[j] that would be used, rejects the call (nothing written at all).  An
 * index value outside [0, in_len[i]) is never dereferenced: that position is
 * not delivered (its destination keeps its value) and the rest is.
 */
BRA_API int indexed_all_to_all_v(const void* const input[], const int64_t in_len[],
                         const int64_t* const index[], const int64_t* send_counts,
                         int64_t* send_displs, int64_t* recv_counts,
                         int64_t* recv_displs, void* const out[], int64_t P,
                         int64_t core_num, int dtype, int32_t* status_dev,
                         bra_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Utilities                                                                 */
/* ------------------------------------------------------------------------ */

/* Human-readable name of a status code (static string, never NULL). */
BRA_API const char* bra_status_str(int status);

/*
 * bra_l2_flush -- read the caller's device buffer `buf` (`bytes` bytes, whole
 * 16-byte words; buf 16-byte aligned) through L2 from a grid-stride kernel on
 * `stream`, so L2 holds clean lines of buf afterwards: data written earlier
 * is back in HBM and written-back before the next timed call, whose inputs
 * then come from HBM (the L2-eviction idea of [VCCL] §7 dev log item D, done
 * with reads so the sweep itself leaves nothing dirty).  Pass a buffer larger
 * than L2.  buf is not modified.
 * Returns BRA_ERR_NULLPTR, BRA_ERR_INVALID (misaligned), BRA_ERR_CUDA or
 * BRA_OK.
 */
BRA_API int bra_l2_flush(void* buf, size_t bytes, bra_stream_t stream);

/*
 * bra_fault_status -- the watchdog words of the current device: 0, or the
 * BRA_ERR_TIMEOUT code a kernel (a tensor-core fused kernel or all_to_all_v) recorded
 * when one of its bounded waits gave up (the kernel then stops early and its
 * output is incomplete).  The words belong to the device, not to a call:
 * every call on the device, on any stream, writes the same words, so a set
 * word says that some call timed out since the last clear, not which.
 * Synchronous (reads device memory after prior work on the legacy stream).
 * With clear != 0 the word is reset to 0.  Returns BRA_OK or BRA_ERR_CUDA.
 */
BRA_API int bra_fault_status(int32_t* code, int clear);

/*
 * bra_wait_selftest -- failure-detection check: launches one kernel whose
 * single bounded wait waits on an mbarrier phase that nothing completes,
 * using the wait helper of the all_to_all_v kernel (which =
 * BRA_WAIT_A2AV, gives up after about 2 s), of the tensor-core fused
 * kernels (BRA_WAIT_TC, about 4 s) or the cluster-scope one of the row-class
 * kernel's MMA issuer (BRA_WAIT_TC_CLUSTER, about 4 s).  The wait runs out,
 * the kernel writes
 * BRA_ERR_TIMEOUT to *status_dev (device int32, BRA_OK had the phase
 * completed), records BRA_ERR_TIMEOUT in the watchdog word that
 * bra_fault_status reads, and returns; nothing traps and the context stays
 * usable.  Asynchronous on `stream`.
 * Returns BRA_ERR_NULLPTR, BRA_ERR_INVALID (unknown `which`), BRA_ERR_CUDA
 * or BRA_OK.
 */
enum { BRA_WAIT_A2AV = 0, BRA_WAIT_TC = 1, BRA_WAIT_TC_CLUSTER = 2 };
BRA_API int bra_wait_selftest(int which, int32_t* status_dev, bra_stream_t stream);

/*
 * bra_mma_rate_probe -- measurement aid for the tensor-core roofline: the
 * dense kind::f16 rate of an SM, measured.  Launches `ctas` CTAs, one per SM
 * (at most the SM count); each issues iters x 4 back-to-back
 * tcgen05.mma.cta_group::1.kind::f16 of M = 128, N = 256, K = 16 (2^20 FLOP
 * each) on zero-filled operands already in shared memory, staged like the
 * fused kernels' (128-byte swizzle, K-major A, N-major B), into one TMEM
 * accumulator, and writes its record to rec_dev[4 * c .. 4 * c + 3] (device
 * int64): SM clock cycles and %globaltimer nanoseconds from the first issue
 * to the completion of the last, BRA_OK or BRA_ERR_TIMEOUT (its bounded
 * wait, about 4 s, ran out), and the SM id.  FLOP per SM clock =
 * iters * 4 * 2^20 / cycles.  dtype: BRA_FP16 or BRA_BF16.  Asynchronous on
 * `stream`.  Returns BRA_ERR_NULLPTR, BRA_ERR_INVALID (ctas outside
 * [1, SM count], iters outside [1, 2^22], other dtype), BRA_ERR_CUDA or
 * BRA_OK.
 */
BRA_API int bra_mma_rate_probe(int ctas, int iters, int dtype, int64_t* rec_dev,
                               bra_stream_t stream);

/*
 * bra_gather_rate_probe -- measurement aid for the indexed exchange's
 * roofline: the rate at which an SM completes random one-byte loads, each in
 * its own 128-byte line (the cost of one gathered element of
 * indexed_all_to_all_v, whose index is arbitrary; [PTO] §A5 URMA 索引交换).
 * Launches `ctas` CTAs of 1024 threads, one per SM (at most the SM count);
 * each thread issues iters x 8 one-byte loads from pseudo-random offsets of
 * buf (device memory of `bytes` bytes, a power of two from 4 KiB to 2^40;
 * only read), and each CTA writes rec_dev[4 * c .. 4 * c + 3] (device int64):
 * SM clock cycles and %globaltimer nanoseconds of its loop, its SM id, and
 * the sum of the bytes it loaded.  Loads per SM clock =
 * 1024 * iters * 8 / cycles.  The loop has no wait.  Asynchronous on
 * `stream`.  Returns BRA_ERR_NULLPTR, BRA_ERR_INVALID (bytes, ctas outside
 * [1, SM count], iters outside [1, 2^20]), BRA_ERR_CUDA or BRA_OK.
 */
BRA_API int bra_gather_rate_probe(const void* buf, int64_t bytes, int ctas, int iters,
                                  int64_t* rec_dev, bra_stream_t stream);

/* Library version, "major.minor.patch". */
BRA_API const char* bra_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BMM_RS_A2A_H */
