"""Oracle for BatchMatMul -> ReduceScatter -> Add -> AllToAll over ep x tp ranks.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition followed ([CANN] §功能说明与计算流程, computation flow):
    temp1 = BatchMatMul(x, weight)
    temp2 = ReduceScatter(temp1)      over the TP group, sum
    temp3 = Add(temp2, bias)
    y     = AllToAll(temp3)           over the EP group
with the transpose needed only for yShardType = 0, the reduce-scatter along H
(dim 2 of the BMM result) for yShardType = 0 and along C (dim 1) for
yShardType = 1 ([CANN] §参数说明, yShardType).

Rank topology ([CANN] §完整调用示例 step 2, EP4 x TP2): rank r = s*tp + t;
EP groups are {t, t+tp, t+2tp, ...} (same t), TP groups {s*tp .. s*tp+tp-1}
(same s).  So s is the rank's EP index and t its TP index.

Readings where the pages are silent:
  * TP-group member t keeps chunk t of the reduce-scatter.
  * The sum runs over t' = 0..tp-1 in index order.  In float64 the order
    moves results only at the 1e-16 level, far below the output rounding.
  * The bias added after the reduce-scatter is the bias of the rank holding
    the reduced chunk (the sender of the all-to-all).
  * AllToAll: chunk j of dim 1 of temp3 goes to EP rank j (rank j*tp + t);
    the receiver stacks what it receives along dim 0 by source EP rank s,
    then local expert e: y[j*tp+t][s*E/ep + e] = chunk j of temp3_{s,t}[e].
  * yShardType = 1 ("blocked" reading): dim 1 of the BMM result, ep*C long,
    is [ep blocks of C tokens] = [ep][tp][C/tp]; TP member t keeps sub-block
    t inside every EP block, so temp2_{s,t}[e, j*C/tp + c'] =
    sum_t' temp1_{s,t'}[e, j*C + t*C/tp + c'].  This is the factorisation the
    guide writes for x's dim 1 (ep*tp*C/tp) and the only reading under which
    the all-to-all delivers EP rank j's own tokens to EP rank j.  The other
    reading ("contiguous": tp plain chunks of the ep*C rows) is kept behind
    `type1_layout` so the tests can show the two are told apart.
  * Products of fp16/bf16 values are exact in float64; sums and the bias add
    are float64 (relative error ~1e-16); one rounding to the output dtype at
    the end.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np

from .rounding import round_to

# Attribute ranges of [CANN] §数据关系与取值范围说明 / §op_api 层; 1 is
# accepted as a degenerate extension for ep and tp.
_WORLD_SIZES = (1, 2, 4, 8, 16, 32)


class OracleParamError(ValueError):
    pass


def check_params(ep, tp, E, C, M, H, y_shard_type) -> None:
    """Range and divisibility rules of [CANN] §数据关系与取值范围说明."""
    if ep not in _WORLD_SIZES or tp not in _WORLD_SIZES:
        raise OracleParamError("ep and tp must be in {1,2,4,8,16,32}")
    if y_shard_type not in (0, 1):
        raise OracleParamError("yShardType must be 0 or 1")
    if not (2 <= E <= 512) or E % ep:
        raise OracleParamError("E must be in [2,512] and a multiple of ep")
    if not (1 <= E // ep <= 32):
        raise OracleParamError("E/ep must be in [1,32]")
    if not (1 <= H <= 65535):
        raise OracleParamError("H must be in [1,65535]")
    if M % tp or not (1 <= M // tp <= 65535):
        raise OracleParamError("M must be a multiple of tp with M/tp in [1,65535]")
    if C <= 0:
        raise OracleParamError("C must be positive")
    if y_shard_type == 0 and H % tp:
        raise OracleParamError("yShardType 0 needs H % tp == 0")
    if y_shard_type == 1 and C % tp:
        raise OracleParamError("yShardType 1 needs C % tp == 0")


def infer_shapes(ep, tp, E, C, M, H, y_shard_type) -> dict:
    """Per-rank shapes, [CANN] §约束说明 and the infershape of §op_api 层:
    yShardType 0 -> y (E, C, H/tp); 1 -> y (E, C/tp, H)."""
    check_params(ep, tp, E, C, M, H, y_shard_type)
    El, Kp = E // ep, M // tp
    if y_shard_type == 0:
        return {"x": (El, ep * C, Kp), "w": (El, Kp, H),
                "bias": (El, 1, H // tp), "y": (E, C, H // tp)}
    return {"x": (El, ep * tp * (C // tp), Kp), "w": (El, Kp, H),
            "bias": (El, 1, H), "y": (E, C // tp, H)}


def _f64(a) -> np.ndarray:
    if a is None:
        return None
    if hasattr(a, "detach"):               # a torch tensor on the host
        a = a.detach().to("cpu")
        import torch
        return a.to(torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def _rs_chunk(total: np.ndarray, t: int, ep, tp, C, H, y_shard_type,
              type1_layout: str) -> np.ndarray:
    """Chunk t of the reduce-scatter of `total` (El, ep*C, H)."""
    if y_shard_type == 0:
        Hp = H // tp
        return total[:, :, t * Hp:(t + 1) * Hp]
    Cp = C // tp
    if type1_layout == "blocked":
        rows = [total[:, j * C + t * Cp: j * C + (t + 1) * Cp, :] for j in range(ep)]
        return np.concatenate(rows, axis=1)
    if type1_layout == "contiguous":
        n = ep * C // tp
        return total[:, t * n:(t + 1) * n, :]
    raise ValueError(type1_layout)


def bmm_rs_a2a(x: Sequence, w: Sequence, bias: Optional[Sequence],
               ep: int, tp: int, E: int, C: int, M: int, H: int,
               y_shard_type: int, dtype: str,
               type1_layout: str = "blocked") -> List[np.ndarray]:
    """Sender view: the four steps of [CANN] §功能说明与计算流程 in order.

    x[r], w[r], bias[r] (r = s*tp + t) are per-rank arrays of the shapes in
    `infer_shapes` (bias may be None, or have the 2-D shape (E/ep, H') of
    [CANN] §参数说明).  Returns y[r] as float64 arrays holding values exactly
    representable in `dtype` ("fp16" | "bf16").  Works one TP group at a time.
    """
    shapes = infer_shapes(ep, tp, E, C, M, H, y_shard_type)
    P = ep * tp
    El = E // ep
    assert len(x) == P and len(w) == P
    y = [np.zeros(shapes["y"], dtype=np.float64) for _ in range(P)]
    # rows of dim 1 of temp3 that form one all-to-all chunk
    chunk_rows = C if y_shard_type == 0 else C // tp
    for s in range(ep):
        # 1. BatchMatMul on each rank of TP group s (float64, exact products).
        temp1 = []
        for t in range(tp):
            r = s * tp + t
            xr, wr = _f64(x[r]), _f64(w[r])
            assert xr.shape == shapes["x"] and wr.shape == shapes["w"]
            temp1.append(np.matmul(xr, wr))              # (El, ep*C, H)
        # 2. ReduceScatter over the TP group: sum in t order, keep chunk t.
        total = temp1[0].copy()
        for t in range(1, tp):
            total += temp1[t]
        for t in range(tp):
            r = s * tp + t
            temp2 = _rs_chunk(total, t, ep, tp, C, H, y_shard_type, type1_layout)
            # 3. Add the bias of this rank, broadcast over dim 1.
            if bias is not None and bias[r] is not None:
                b = _f64(bias[r]).reshape(El, 1, -1)
                temp3 = temp2 + b
            else:
                temp3 = temp2
            # 4. AllToAll over the EP group: chunk j of dim 1 -> EP rank j,
            #    stacked at dim-0 block s*El .. s*El+El-1 of the receiver.
            for j in range(ep):
                d = j * tp + t
                y[d][s * El:(s + 1) * El] = temp3[:, j * chunk_rows:(j + 1) * chunk_rows, :]
    return [round_to(a, dtype) for a in y]


def group_outputs(x_group: Sequence, w_group: Sequence, bias_group: Optional[Sequence],
                  ep: int, tp: int, C: int, H: int, y_shard_type: int, dtype: str,
                  type1_layout: str = "blocked") -> dict:
    """Sender view for one TP group s and one local expert e: the four steps
    of [CANN] §功能说明与计算流程 restricted to that (s, e), so that a whole
    expert block of a large problem can be evaluated without the others.

    x_group[t], w_group[t]: expert e of rank s*tp+t, shapes (ep*C, M/tp) and
    (M/tp, H); bias_group: None, or tp rows (length H/tp for yShardType 0, H
    for 1) holding expert e's bias of rank s*tp+t.  Returns {(j, t): block},
    the block receiver j*tp+t stores at dim-0 index s*E/ep + e (shape (C,
    H/tp) for yShardType 0, (C/tp, H) for 1), as float64 arrays of values
    exactly representable in `dtype`.
    """
    assert len(x_group) == tp and len(w_group) == tp
    # 1. BatchMatMul on every rank of the group, 2. summed in t order.
    total = None
    for t in range(tp):
        prod = np.matmul(_f64(x_group[t]), _f64(w_group[t]))   # (ep*C, H)
        total = prod if total is None else total + prod
    chunk_rows = C if y_shard_type == 0 else C // tp
    out = {}
    for t in range(tp):
        temp2 = _rs_chunk(total[None], t, ep, tp, C, H, y_shard_type, type1_layout)[0]
        # 3. this rank's bias, broadcast over the rows
        temp3 = temp2 if bias_group is None else temp2 + _f64(bias_group[t]).reshape(1, -1)
        # 4. chunk j of the rows goes to EP rank j
        for j in range(ep):
            out[(j, t)] = round_to(temp3[j * chunk_rows:(j + 1) * chunk_rows], dtype)
    return out


def y_source(ep, tp, E, C, H, y_shard_type, d, i, c, h,
             type1_layout: str = "blocked") -> dict:
    """Receiver view: where output element y[d][i, c, h] comes from.

    Returns the sending rank's EP index s and TP index t, the local expert e,
    the row and column of the tp-summed BMM result Z_{s,e} = sum_t'
    x[s*tp+t'][e] @ w[s*tp+t'][e] (shape (ep*C, H)), and the bias position.
    """
    El = E // ep
    j, t = divmod(d, tp)          # receiving rank's EP and TP index
    s, e = divmod(i, El)          # stacked by source EP rank, then expert
    if y_shard_type == 0:
        zrow = j * C + c
        zcol = t * (H // tp) + h
    else:
        Cp = C // tp
        if type1_layout == "blocked":
            zrow = j * C + t * Cp + c
        else:
            zrow = t * (ep * C // tp) + j * Cp + c
        zcol = h
    return {"s": s, "t": t, "e": e, "zrow": zrow, "zcol": zcol,
            "bias_rank": s * tp + t, "bias_col": h}


def bmm_rs_a2a_point(x_rows: np.ndarray, w_cols: np.ndarray,
                     bias_value: Optional[float], dtype: str) -> float:
    """One output value: sum over t' of the dot product of row zrow of
    x[s*tp+t'][e] with column zcol of w[s*tp+t'][e], plus the bias, rounded.

    x_rows, w_cols: (tp, M/tp) float arrays, row t' belonging to rank s*tp+t'.
    """
    x_rows = np.asarray(x_rows, dtype=np.float64)
    w_cols = np.asarray(w_cols, dtype=np.float64)
    acc = 0.0
    for tt in range(x_rows.shape[0]):
        acc += float(np.dot(x_rows[tt], w_cols[tt]))
    if bias_value is not None:
        acc += float(bias_value)
    return float(round_to(np.array([acc]), dtype)[0])


def naive_bmm_rs_a2a(x, w, bias, ep, tp, E, C, M, H, y_shard_type, dtype,
                     type1_layout: str = "blocked") -> List[np.ndarray]:
    """Receiver view with scalar Python loops; only for tiny shapes."""
    shapes = infer_shapes(ep, tp, E, C, M, H, y_shard_type)
    P = ep * tp
    xs = [_f64(a) for a in x]
    ws = [_f64(a) for a in w]
    bs = None if bias is None else [None if b is None else _f64(b).reshape(E // ep, -1)
                                    for b in bias]
    Kp = M // tp
    out = []
    for d in range(P):
        yd = np.zeros(shapes["y"], dtype=np.float64)
        n0, n1, n2 = shapes["y"]
        for i in range(n0):
            for c in range(n1):
                for h in range(n2):
                    src = y_source(ep, tp, E, C, H, y_shard_type, d, i, c, h, type1_layout)
                    acc = 0.0
                    for tt in range(tp):
                        r = src["s"] * tp + tt
                        for k in range(Kp):
                            acc += xs[r][src["e"], src["zrow"], k] * ws[r][src["e"], k, src["zcol"]]
                    if bs is not None and bs[src["bias_rank"]] is not None:
                        acc += bs[src["bias_rank"]][src["e"], src["bias_col"]]
                    yd[i, c, h] = acc
        out.append(round_to(yd, dtype))
    return out
