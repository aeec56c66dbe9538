"""Oracle for all_to_all_v and its launch-width rule.

TEST INFRASTRUCTURE ONLY (see the package docstring).

all_to_all_v ([PTO] §行为 and §ABI; [VCCL] §5 ref, the meta ncclx alltoallv
addressing): rank i sends send_counts[i][j] elements to rank j.  Rank i's
elements for rank j start at its send displacement, the ones it receives from
rank i land at its receive displacement; displacements are exclusive prefix
sums in element units, the sender's over destinations and the receiver's over
sources, so rank j's output holds what it received ordered by source rank.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np

INT32_MAX = 2**31 - 1


def cal_all_to_all_v_blocks(P: int, L: int) -> int:
    """Admitted block count B ([PTO] §启动宽度, launch width): L when L < P,
    otherwise the largest multiple of P not above L.  Returns -1 for P < 1 or
    L outside [1, INT32_MAX] ([PTO] §约束与诊断)."""
    if P < 1 or L < 1 or L > INT32_MAX:
        return -1
    if L < P:
        return L
    return (L // P) * P


def a2av_bookkeeping(send_counts: np.ndarray):
    """(send_displs, recv_counts, recv_displs), each P x P int64.

    send_displs[i][j] = sum_{k<j} send_counts[i][k]
    recv_counts[j][i] = send_counts[i][j]
    recv_displs[j][i] = sum_{k<i} send_counts[k][j]
    """
    sc = np.asarray(send_counts, dtype=np.int64)
    P = sc.shape[0]
    assert sc.shape == (P, P)
    sd = np.zeros((P, P), dtype=np.int64)
    rc = np.zeros((P, P), dtype=np.int64)
    rd = np.zeros((P, P), dtype=np.int64)
    for i in range(P):
        run = 0
        for j in range(P):
            sd[i, j] = run
            run += int(sc[i, j])
    for j in range(P):
        run = 0
        for i in range(P):
            rc[j, i] = sc[i, j]
            rd[j, i] = run
            run += int(sc[i, j])
    return sd, rc, rd


def all_to_all_v(inputs: Sequence[np.ndarray], send_counts: np.ndarray,
                 out_init: Sequence[np.ndarray]) -> dict:
    """Exchange: out[j][rd[j][i] : rd[j][i]+n] = inputs[i][sd[i][j] : sd[i][j]+n]
    with n = send_counts[i][j], for every pair (i, j) including i == j.

    out_init[j] is rank j's output buffer before the call (copied, not
    modified); elements past what rank j receives keep their initial value.
    Negative counts are rejected (the whole call does nothing), matching the
    count-matrix categories the [PTO] §测试 system test exercises.
    """
    sc = np.asarray(send_counts, dtype=np.int64)
    P = sc.shape[0]
    if (sc < 0).any():
        raise ValueError("negative send count")
    sd, rc, rd = a2av_bookkeeping(sc)
    out: List[np.ndarray] = [np.array(o, copy=True) for o in out_init]
    for i in range(P):
        src = inputs[i]
        for j in range(P):
            n = int(sc[i, j])
            if n == 0:
                continue
            a, b = int(sd[i, j]), int(rd[j, i])
            if a + n > len(src) or b + n > len(out[j]):
                raise ValueError(f"pair ({i},{j}) exceeds a buffer")
            out[j][b:b + n] = src[a:a + n]
    return {"out": out, "send_displs": sd, "recv_counts": rc, "recv_displs": rd}


def received_totals(send_counts: np.ndarray) -> np.ndarray:
    """Elements rank j receives, summed pair by pair."""
    sc = np.asarray(send_counts, dtype=np.int64)
    P = sc.shape[0]
    tot = np.zeros(P, dtype=np.int64)
    for i in range(P):
        for j in range(P):
            tot[j] += sc[i, j]
    return tot


def indexed_all_to_all_v(inputs: Sequence[np.ndarray], index: Sequence[np.ndarray],
                         send_counts: np.ndarray, out_init: Sequence[np.ndarray]) -> dict:
    """Indexed exchange ([PTO] §A5 URMA 索引交换): the page names the operands
    (input, send_counts, recv_counts, index) and says the cores share the
    local data movement before the remote transfers; it does not define
    `index`.  Reading taken here: the local movement gathers rank i's send
    list from its input through its index, then the send lists are exchanged
    as in all_to_all_v:

        send_i[k] = inputs[i][index[i][k]]        k < sum_j send_counts[i][j]
        out[j][rd[j][i] + m] = send_i[sd[i][j] + m]   m < send_counts[i][j]

    An index value outside [0, len(inputs[i])) is an error: that element is
    not delivered (its destination keeps the initial value) and is counted in
    "invalid".  Negative counts reject the whole call, as in all_to_all_v.
    """
    sc = np.asarray(send_counts, dtype=np.int64)
    P = sc.shape[0]
    if (sc < 0).any():
        raise ValueError("negative send count")
    sd, rc, rd = a2av_bookkeeping(sc)
    out: List[np.ndarray] = [np.array(o, copy=True) for o in out_init]
    invalid = 0
    for i in range(P):
        src = np.asarray(inputs[i])
        idx = np.asarray(index[i], dtype=np.int64)
        n = int(sc[i].sum())
        if len(idx) < n:
            raise ValueError(f"rank {i}: index shorter than its send list")
        # local movement: the send list and which of its entries exist
        ok = (idx[:n] >= 0) & (idx[:n] < len(src))
        invalid += int((~ok).sum())
        send = np.zeros(n, dtype=src.dtype)
        send[ok] = src[idx[:n][ok]]
        # the exchange of the send list
        for j in range(P):
            c = int(sc[i, j])
            if c == 0:
                continue
            a, b = int(sd[i, j]), int(rd[j, i])
            if b + c > len(out[j]):
                raise ValueError(f"pair ({i},{j}) exceeds a buffer")
            keep = ok[a:a + c]
            out[j][b:b + c][keep] = send[a:a + c][keep]
    return {"out": out, "send_displs": sd, "recv_counts": rc, "recv_displs": rd,
            "invalid": invalid}
