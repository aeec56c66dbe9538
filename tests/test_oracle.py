"""Pins for the CPU oracle: each test ties it to something other than itself.

CPU only.  A plausible mistake in the oracle (a dropped tp term, a wrong chunk
index, a transposed operand, the wrong bias owner, a wrong prefix sum, a
wrong launch-width rule) fails at least one of these.
"""
import itertools
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import a2av as oa
from oracle import fused as of
from oracle.rounding import round_bf16, round_fp16
from workloads import A2AVConfig, FusedConfig, a2av_inputs, fused_inputs_host

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


# --------------------------------------------------------------------------
# CalAllToAllVBlocks
# --------------------------------------------------------------------------

def test_cal_blocks_golden_table():
    rows = list(_rows("cal_all_to_all_v_blocks.txt"))
    assert any(r.endswith("printed") for r in rows)
    for r in rows:
        P, L, B, _ = r.split()
        assert oa.cal_all_to_all_v_blocks(int(P), int(L)) == int(B), r


def test_cal_blocks_is_largest_admissible_count():
    # Characterisation: B is the largest b <= L that is either below P or a
    # multiple of P (the counts a block-aware barrier over P peers admits).
    for P in range(1, 34):
        for L in range(1, 140):
            admissible = [b for b in range(1, L + 1) if b < P or b % P == 0]
            assert oa.cal_all_to_all_v_blocks(P, L) == max(admissible)


def test_signal_stride_example():
    # The page: L=10, P=8 launches 8 blocks, so a signal stride S=8 passes S >= B.
    assert 8 >= oa.cal_all_to_all_v_blocks(8, 10)
    assert not (8 >= oa.cal_all_to_all_v_blocks(8, 16))


# --------------------------------------------------------------------------
# all_to_all_v
# --------------------------------------------------------------------------

def _a2av_case(P, seed, hi=7, zero_frac=0.3):
    rng = np.random.default_rng(seed)
    sc = rng.integers(0, hi + 1, size=(P, P)).astype(np.int64)
    sc[rng.random((P, P)) < zero_frac] = 0
    inputs = [rng.standard_normal(int(sc[i].sum())) for i in range(P)]
    return sc, inputs


def test_bookkeeping_matches_cumsum():
    for P in (1, 2, 3, 8, 32):
        sc, _ = _a2av_case(P, seed=P)
        sd, rc, rd = oa.a2av_bookkeeping(sc)
        z = np.zeros((P, 1), dtype=np.int64)
        np.testing.assert_array_equal(sd, np.hstack([z, np.cumsum(sc, axis=1)[:, :-1]]))
        np.testing.assert_array_equal(rc, sc.T)
        np.testing.assert_array_equal(rd, np.hstack([z, np.cumsum(sc.T, axis=1)[:, :-1]]))


def test_exchange_with_transposed_counts_inverts_itself():
    for P in (1, 2, 3, 5, 8):
        sc, inputs = _a2av_case(P, seed=10 + P)
        tot = sc.sum(axis=0)
        first = oa.all_to_all_v(inputs, sc, [np.zeros(int(n)) for n in tot])["out"]
        back = oa.all_to_all_v(first, sc.T.copy(),
                               [np.zeros(len(a)) for a in inputs])["out"]
        for a, b in zip(inputs, back):
            np.testing.assert_array_equal(a, b)


def test_received_totals_are_column_sums_and_tail_untouched():
    sentinel = -12345.0
    for P in (2, 4, 8):
        sc, inputs = _a2av_case(P, seed=20 + P)
        cols = sc.sum(axis=0)
        np.testing.assert_array_equal(oa.received_totals(sc), cols)
        init = [np.full(int(n) + 5, sentinel) for n in cols]
        out = oa.all_to_all_v(inputs, sc, init)["out"]
        for j in range(P):
            assert (out[j][int(cols[j]):] == sentinel).all()
            assert not (out[j][:int(cols[j])] == sentinel).any()


def test_exchange_brute_force_by_tags():
    # Tag every element with (source, destination, ordinal); the receiver must
    # hold, source by source in rank order, exactly the tags addressed to it.
    for P, seed in itertools.product((1, 2, 3, 4), range(4)):
        rng = np.random.default_rng(100 + seed)
        sc = rng.integers(0, 4, size=(P, P)).astype(np.int64)
        tags = []
        for i in range(P):
            row = []
            for j in range(P):
                row += [(i, j, k) for k in range(int(sc[i, j]))]
            tags.append(row)
        enc = [np.array([a * 10000 + b * 100 + c for a, b, c in row], dtype=np.float64)
               for row in tags]
        cols = sc.sum(axis=0)
        out = oa.all_to_all_v(enc, sc, [np.zeros(int(n)) for n in cols])["out"]
        for j in range(P):
            expect = [i * 10000 + j * 100 + k for i in range(P) for k in range(int(sc[i, j]))]
            np.testing.assert_array_equal(out[j], np.array(expect, dtype=np.float64))


# --------------------------------------------------------------------------
# indexed all_to_all_v (reading: gather through the index, then exchange)
# --------------------------------------------------------------------------

def _indexed_case(P, seed, hi=5, extra=3):
    rng = np.random.default_rng(seed)
    sc = rng.integers(0, hi + 1, size=(P, P)).astype(np.int64)
    lens = [int(sc[i].sum()) + int(rng.integers(0, extra + 1)) for i in range(P)]
    inputs = [rng.standard_normal(n) for n in lens]
    index = [rng.integers(0, max(n, 1), size=int(sc[i].sum())) for i, n in enumerate(lens)]
    return sc, inputs, index


def test_indexed_with_identity_index_is_all_to_all_v():
    for P in (1, 2, 3, 8):
        sc, inputs = _a2av_case(P, seed=40 + P)
        cols = sc.sum(axis=0)
        init = [np.full(int(n) + 2, -7.0) for n in cols]
        ident = [np.arange(len(a), dtype=np.int64) for a in inputs]
        a = oa.all_to_all_v(inputs, sc, init)
        b = oa.indexed_all_to_all_v(inputs, ident, sc, init)
        assert b["invalid"] == 0
        for u, v in zip(a["out"], b["out"]):
            np.testing.assert_array_equal(u, v)
        for k in ("send_displs", "recv_counts", "recv_displs"):
            np.testing.assert_array_equal(a[k], b[k])


def test_indexed_brute_force_by_tags():
    # Input element p of rank i carries the tag i * 1000 + p.  Walking each
    # sender's destinations in rank order with a running position, the m-th
    # element rank j receives from rank i must carry the tag of the input
    # element that rank i's index names at that position.
    for P, seed in itertools.product((1, 2, 3, 4), range(4)):
        sc, inputs, index = _indexed_case(P, seed=200 + 10 * P + seed)
        tagged = [np.array([i * 1000 + q for q in range(len(inputs[i]))], dtype=np.float64)
                  for i in range(P)]
        expect = [[] for _ in range(P)]
        for j in range(P):
            for i in range(P):
                pos = 0
                for jj in range(P):
                    for m in range(int(sc[i, jj])):
                        if jj == j:
                            expect[j].append(i * 1000 + int(index[i][pos]))
                        pos += 1
        cols = sc.sum(axis=0)
        out = oa.indexed_all_to_all_v(tagged, index, sc, [np.zeros(int(n)) for n in cols])["out"]
        for j in range(P):
            np.testing.assert_array_equal(out[j], np.array(expect[j], dtype=np.float64))


def test_indexed_permutation_conserves_the_elements():
    for P in (2, 5, 8):
        rng = np.random.default_rng(300 + P)
        sc = rng.integers(0, 9, size=(P, P)).astype(np.int64)
        inputs = [rng.standard_normal(int(sc[i].sum())) for i in range(P)]
        index = [rng.permutation(len(a)) for a in inputs]
        cols = sc.sum(axis=0)
        r = oa.indexed_all_to_all_v(inputs, index, sc, [np.zeros(int(n)) for n in cols])
        assert r["invalid"] == 0
        np.testing.assert_array_equal(np.sort(np.concatenate(r["out"])),
                                      np.sort(np.concatenate(inputs)))


def test_indexed_out_of_range_not_delivered_and_counted():
    sc = np.array([[2, 1], [1, 2]], dtype=np.int64)
    inputs = [np.array([10.0, 11.0, 12.0]), np.array([20.0, 21.0, 22.0, 23.0])]
    index = [np.array([2, -1, 0]), np.array([4, 1, 3])]   # -1 and 4 are outside
    init = [np.full(3, -5.0), np.full(3, -5.0)]
    r = oa.indexed_all_to_all_v(inputs, index, sc, init)
    assert r["invalid"] == 2
    np.testing.assert_array_equal(r["out"][0], [12.0, -5.0, -5.0])   # from 0: 12, bad; from 1: bad
    np.testing.assert_array_equal(r["out"][1], [10.0, 21.0, 23.0])
    with pytest.raises(ValueError):
        oa.indexed_all_to_all_v(inputs, index, np.array([[1, -1], [0, 1]]), init)


def test_negative_counts_rejected():
    sc = np.array([[1, -1], [0, 2]], dtype=np.int64)
    with pytest.raises(ValueError):
        oa.all_to_all_v([np.zeros(1), np.zeros(2)], sc, [np.zeros(4), np.zeros(4)])


def test_workload_generators_shape_the_counts():
    c2 = A2AVConfig("u", P=8, L=10, dtype="fp32", seed=1, counts="uniform")
    sc, inp = a2av_inputs(c2)
    assert sc.shape == (8, 8) and sc.min() >= 0 and sc.max() <= 4096
    assert [len(a) for a in inp] == list(sc.sum(axis=1))
    c4 = A2AVConfig("d", P=32, L=64, dtype="int8", seed=3, counts="dirichlet")
    sc4, inp4 = a2av_inputs(c4)
    assert (sc4 == 0).any()                       # zero-count pairs present
    per_rank = sc4.sum(axis=1)
    assert abs(per_rank.mean() - 2**21) < 64      # ~2 MiB sent per rank
    assert inp4[0].dtype == np.int8


# --------------------------------------------------------------------------
# Fused op: shapes and checks
# --------------------------------------------------------------------------

def test_shapes_of_the_guides_example():
    for r in _rows("shapes_ep4_tp2_example.txt"):
        head, xs, ws, bs, ys = [p.split() for p in r.split("|")]
        ep, tp, E, C, M, H, t = map(int, head)
        sh = of.infer_shapes(ep, tp, E, C, M, H, t)
        assert sh["x"] == tuple(map(int, xs))
        assert sh["w"] == tuple(map(int, ws))
        assert sh["bias"] == tuple(map(int, bs))
        assert sh["y"] == tuple(map(int, ys))


def test_shape_relations_of_the_dim_checks():
    # CheckTensorDimCommonShape / CheckTensorDimUniqueShape relations.
    for ep, tp in itertools.product((1, 2, 4, 8), (1, 2, 4)):
        for t in (0, 1):
            E, C, M, H = 8 * ep, 4 * tp, 8 * tp, 6 * tp
            sh = of.infer_shapes(ep, tp, E, C, M, H, t)
            x, w, y = sh["x"], sh["w"], sh["y"]
            assert y[0] == x[0] * ep and x[0] == w[0] and x[2] == w[1]
            if t == 0:
                assert w[2] == y[2] * tp and x[1] == y[1] * ep
            else:
                assert w[2] == y[2] and x[1] == y[1] * ep * tp


@pytest.mark.parametrize("bad", [
    dict(ep=3), dict(tp=64), dict(E=1), dict(E=514), dict(E=20, ep=8),
    dict(E=264, ep=8), dict(H=65536), dict(M=2 * 65536), dict(C=0),
    dict(H=5, t=0), dict(C=5, t=1), dict(t=2)])
def test_parameter_ranges(bad):
    p = dict(ep=2, tp=2, E=8, C=4, M=8, H=8, t=0)
    p.update(bad)
    with pytest.raises(of.OracleParamError):
        of.infer_shapes(p["ep"], p["tp"], p["E"], p["C"], p["M"], p["H"], p["t"])


# --------------------------------------------------------------------------
# Fused op: values
# --------------------------------------------------------------------------

def _cfg(ep, tp, E, C, M, H, t, dtype="fp16", seed=0, bias=True):
    return FusedConfig("t", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t,
                       dtype=dtype, seed=seed, has_bias=bias)


def _run(cfg, inp, **kw):
    return of.bmm_rs_a2a(inp["x"], inp["w"], inp["bias"], cfg.ep, cfg.tp, cfg.E,
                         cfg.C, cfg.M, cfg.H, cfg.y_shard_type, cfg.dtype, **kw)


def _np(t):
    return None if t is None else t.to(torch.float64).numpy()


@pytest.mark.parametrize("t", [0, 1])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_ep1_tp1_is_a_batched_matmul_plus_bias(t, dtype):
    cfg = _cfg(1, 1, 3, 5, 7, 6, t, dtype)
    inp = fused_inputs_host(cfg)
    y = _run(cfg, inp)[0]
    x, w, b = _np(inp["x"][0]), _np(inp["w"][0]), _np(inp["bias"][0])
    ref = np.einsum("ecm,emh->ech", x, w) + b
    rnd = round_fp16 if dtype == "fp16" else round_bf16
    np.testing.assert_array_equal(y, rnd(ref))


@pytest.mark.parametrize("t", [0, 1])
def test_tp1_is_a_permuted_bmm(t):
    ep, E, C, M, H = 4, 8, 3, 5, 6
    cfg = _cfg(ep, 1, E, C, M, H, t, seed=3)
    inp = fused_inputs_host(cfg)
    y = _run(cfg, inp)
    X = np.stack([_np(a) for a in inp["x"]])          # (s, e, ep*C, M)
    W = np.stack([_np(a) for a in inp["w"]])          # (s, e, M, H)
    B = np.stack([_np(a) for a in inp["bias"]])       # (s, e, 1, H)
    Z = np.einsum("secm,semh->sech", X, W) + B        # (s, e, ep*C, H)
    El = E // ep
    for j in range(ep):
        # receiver j: block (s, e) = rows j*C..j*C+C-1 of sender s's expert e
        ref = Z[:, :, j * C:(j + 1) * C, :].reshape(ep * El, C, H)
        np.testing.assert_array_equal(y[j], round_fp16(ref))


@pytest.mark.parametrize("ep,tp", [(2, 2), (2, 4), (4, 2), (1, 4)])
@pytest.mark.parametrize("t", [0, 1])
def test_tp_reduction_is_one_matmul_over_concatenated_contraction(ep, tp, t):
    # sum_t x_t @ w_t == [x_0 | x_1 | ...] @ [w_0 ; w_1 ; ...]: compare the
    # tp-way op (no bias) with the tp=1 op on K-concatenated operands.
    E, C, M, H = 2 * ep, 2 * tp, 3 * tp, 2 * tp
    cfg = _cfg(ep, tp, E, C, M, H, t, seed=7, bias=False)
    inp = fused_inputs_host(cfg)
    y = _run(cfg, inp)
    xc = [np.concatenate([_np(inp["x"][s * tp + u]) for u in range(tp)], axis=2) for s in range(ep)]
    wc = [np.concatenate([_np(inp["w"][s * tp + u]) for u in range(tp)], axis=1) for s in range(ep)]
    y1 = of.bmm_rs_a2a(xc, wc, None, ep, 1, E, C, M, H, 0, "fp16")
    Hp, Cp = H // tp, C // tp
    for j in range(ep):
        for u in range(tp):
            if t == 0:
                ref = y1[j][:, :, u * Hp:(u + 1) * Hp]
            else:
                ref = y1[j][:, u * Cp:(u + 1) * Cp, :]
            np.testing.assert_array_equal(y[j * tp + u], ref)


def test_bias_belongs_to_the_sender():
    ep, tp, E, C, M, H = 4, 2, 8, 4, 4, 4
    for t in (0, 1):
        cfg = _cfg(ep, tp, E, C, M, H, t)
        inp = fused_inputs_host(cfg)
        inp["x"] = [torch.zeros_like(a) for a in inp["x"]]
        inp["bias"] = [torch.full_like(b, float(r + 1)) for r, b in enumerate(inp["bias"])]
        y = _run(cfg, inp)
        El = E // ep
        for d in range(ep * tp):
            u = d % tp
            for s in range(ep):
                assert (y[d][s * El:(s + 1) * El] == s * tp + u + 1).all()


def test_type1_delivers_each_ep_rank_its_own_tokens():
    # Token tags: x[..., m, 0] = m + 1 and weight row 0 = 1, so each output
    # row carries the BMM row it came from (summed over the tp shards).
    ep, tp, E, C, M, H = 4, 2, 8, 8, 4, 3
    cfg = _cfg(ep, tp, E, C, M, H, 1, bias=False)
    inp = fused_inputs_host(cfg)
    for a in inp["x"]:
        a.zero_()
        a[:, :, 0] = torch.arange(1, a.shape[1] + 1, dtype=a.dtype)
    for a in inp["w"]:
        a.zero_()
        a[:, 0, :] = 1
    got = {}
    for layout in ("blocked", "contiguous"):
        y = _run(cfg, inp, type1_layout=layout)
        ok = True
        for d in range(ep * tp):
            j = d // tp
            rows = y[d][..., 0] / tp - 1            # tp shards each add m+1
            ok &= bool(((rows >= j * C) & (rows < (j + 1) * C)).all())
        got[layout] = ok
    assert got == {"blocked": True, "contiguous": False}


@pytest.mark.parametrize("ep,tp", list(itertools.product((1, 2, 4), (1, 2, 4))))
@pytest.mark.parametrize("t", [0, 1])
@pytest.mark.parametrize("bias_ndim", [0, 2, 3])
def test_sender_view_equals_receiver_view_brute_force(ep, tp, t, bias_ndim):
    E, C, M, H = 2 * ep, 2 * tp, 3 * tp, 2 * tp
    dtype = "bf16" if (ep + tp + t) % 2 else "fp16"
    cfg = _cfg(ep, tp, E, C, M, H, t, dtype=dtype, seed=ep * 10 + tp, bias=bias_ndim > 0)
    inp = fused_inputs_host(cfg, bias_ndim=bias_ndim or 3)
    a = _run(cfg, inp)
    b = of.naive_bmm_rs_a2a(inp["x"], inp["w"], inp["bias"], ep, tp, E, C, M, H, t, dtype)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


@pytest.mark.parametrize("ep,tp", [(1, 1), (2, 2), (4, 2), (2, 4)])
@pytest.mark.parametrize("t", [0, 1])
@pytest.mark.parametrize("bias", [True, False])
@pytest.mark.parametrize("layout", ["blocked", "contiguous"])
def test_group_outputs_are_the_full_oracles_blocks(ep, tp, t, bias, layout):
    """One (s, e) evaluated alone gives exactly the blocks the whole-problem
    oracle writes for it, at every receiver (both type-1 readings)."""
    E, C, M, H = 3 * ep, 3 * tp, 5 * tp, 2 * tp
    cfg = _cfg(ep, tp, E, C, M, H, t, dtype="bf16" if t else "fp16", seed=ep + 3 * tp,
               bias=bias)
    inp = fused_inputs_host(cfg)
    y = _run(cfg, inp, type1_layout=layout)
    El = E // ep
    for s in range(ep):
        for e in range(El):
            rs = [s * tp + u for u in range(tp)]
            bg = None if not bias else [inp["bias"][r].reshape(El, -1)[e] for r in rs]
            blocks = of.group_outputs([inp["x"][r][e] for r in rs], [inp["w"][r][e] for r in rs],
                                      bg, ep, tp, C, H, t, cfg.dtype, type1_layout=layout)
            assert sorted(blocks) == [(j, u) for j in range(ep) for u in range(tp)]
            for (j, u), blk in blocks.items():
                np.testing.assert_array_equal(blk, y[j * tp + u][s * El + e])


def test_group_outputs_brute_force():
    """Against the receiver-view scalar loops on a tiny problem."""
    ep, tp, E, C, M, H = 2, 2, 4, 4, 6, 4
    for t in (0, 1):
        cfg = _cfg(ep, tp, E, C, M, H, t, seed=11 + t)
        inp = fused_inputs_host(cfg)
        ref = of.naive_bmm_rs_a2a(inp["x"], inp["w"], inp["bias"], ep, tp, E, C, M, H, t,
                                  "fp16")
        for s in range(ep):
            for e in range(E // ep):
                rs = [s * tp + u for u in range(tp)]
                blocks = of.group_outputs([inp["x"][r][e] for r in rs],
                                          [inp["w"][r][e] for r in rs],
                                          [inp["bias"][r][e, 0] for r in rs],
                                          ep, tp, C, H, t, "fp16")
                for (j, u), blk in blocks.items():
                    np.testing.assert_array_equal(blk, ref[j * tp + u][s * (E // ep) + e])


def test_point_evaluation_matches_full_oracle():
    cfg = _cfg(4, 2, 16, 12, 12, 4, 1)
    inp = fused_inputs_host(cfg)
    y = _run(cfg, inp)
    rng = np.random.default_rng(5)
    xs = [_np(a) for a in inp["x"]]
    ws = [_np(a) for a in inp["w"]]
    bs = [_np(b).reshape(4, -1) for b in inp["bias"]]
    for _ in range(200):
        d = int(rng.integers(8))
        i, c, h = (int(rng.integers(n)) for n in y[d].shape)
        src = of.y_source(4, 2, 16, 12, 4, 1, d, i, c, h)
        rows = np.stack([xs[src["s"] * 2 + u][src["e"], src["zrow"], :] for u in range(2)])
        cols = np.stack([ws[src["s"] * 2 + u][src["e"], :, src["zcol"]] for u in range(2)])
        v = of.bmm_rs_a2a_point(rows, cols, bs[src["bias_rank"]][src["e"], src["bias_col"]], "fp16")
        assert v == y[d][i, c, h]


# --------------------------------------------------------------------------
# Rounding
# --------------------------------------------------------------------------

def test_bf16_rounding_equals_torch_on_float32_inputs():
    rng = np.random.default_rng(0)
    with np.errstate(over="ignore"):                                # a few become inf on purpose
        near_overflow = (rng.standard_normal(2000) * 1e38).astype(np.float32)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),     # subnormals
        near_overflow,                                              # near overflow
        np.array([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8), 3.3895314e38, 0.0, -0.0],
                 dtype=np.float32)])
    ours = round_bf16(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_bf16_ties_and_overflow():
    assert round_bf16(np.array([1 + 2**-8]))[0] == 1.0                     # tie -> even
    assert round_bf16(np.array([1 + 3 * 2**-8]))[0] == 1 + 2**-6           # tie -> even
    assert round_bf16(np.array([1 + 2**-8 + 2**-30]))[0] == 1 + 2**-7      # above tie
    assert np.isinf(round_bf16(np.array([2.0**128]))[0])
    assert round_bf16(np.array([2.0**-130]))[0] == 2.0**-130                # subnormal exact
    assert round_bf16(np.array([2.0**-134]))[0] == 0.0                      # half the least -> even (0)
    assert round_bf16(np.array([3 * 2.0**-134]))[0] == 2.0**-132            # 1.5 least -> even (2)
    assert round_bf16(np.array([3 * 2.0**-135]))[0] == 2.0**-133            # 0.75 least -> 1


def test_fp16_rounding_ties_and_overflow():
    assert round_fp16(np.array([1 + 2**-11]))[0] == 1.0
    assert round_fp16(np.array([2049.0]))[0] == 2048.0
    assert np.isinf(round_fp16(np.array([65520.0]))[0])
    assert round_fp16(np.array([65519.0]))[0] == 65504.0
