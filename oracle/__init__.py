"""CPU oracle for the fused BMM-RS-Add-A2A op and for all_to_all_v.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the pages define, evaluated in float64 (integers exact)
with a single final rounding to the output dtype.  Only the test-suite, the
smoke check of `__graft_entry__` and the CPU-baseline leg of `bench.py` may
import it; the product library never does, and the oracle imports nothing from
the product (it shares no code, header, table or helper with the CUDA path).

Sources (pages, cited by title and section):
  [CANN] "CANN ops-transformer 通算融合算子实战 BatchMatMulReduceScatterAllToAll
         原理、shape 约束与 aclnn 两段式调用" (pnsm.cn)
  [PTO]  "LowerL2TensorCollectives Pass" (pypto.ai)
  [VCCL] "vccl alltoallv dev log" (obnotes)

Modules:
  fused     -- infer_shapes, bmm_rs_a2a (sender view, the four steps in order),
               y_source / bmm_rs_a2a_point (receiver view, per element)
  a2av      -- cal_all_to_all_v_blocks, a2av_bookkeeping, all_to_all_v,
               indexed_all_to_all_v (gather through the index, then exchange)
  rounding  -- float64 -> fp16 / bf16 round-to-nearest-even

Pins (tests/test_oracle.py): the printed CalAllToAllVBlocks example and rule
table, the shape relations, ep=tp=1 reducing to a textbook batched matmul plus
bias, tp=1 reducing to a permuted BMM (einsum), the tp reduction equalling one
matmul over the concatenated contraction dimension, the exchange inverting
itself under transposed counts, received totals equalling column sums, the
bookkeeping equalling numpy's cumsum, bf16 rounding equalling torch's, and the
two independent formulations (sender and receiver view) agreeing on tiny
inputs.  The yShardType=1 row layout is pinned to the reading stated in
`fused` (the pages fix only the shape), and tests show the alternative reading
is distinguishable.
"""
from . import a2av, fused, rounding  # noqa: F401
from .a2av import a2av_bookkeeping, all_to_all_v, cal_all_to_all_v_blocks  # noqa: F401
from .fused import (bmm_rs_a2a, bmm_rs_a2a_point, infer_shapes,  # noqa: F401
                    y_source)
