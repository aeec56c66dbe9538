"""indexed_all_to_all_v on the GPU against the CPU oracle: bit-exact.

Reading under test (the URMA indexed exchange of the PyPTO page): each
sender's list is its input gathered through its index, then exchanged as in
all_to_all_v.  Covers identity, permutation and repeating indices over
longer inputs, fp32 and int8, P from 1 to 64, the int8 P = 32 Dirichlet
workload at full size, unaligned input and output views, out-of-range index
values (not delivered, reported), the device-side rejections (negative
count, a NULL buffer that would be used: nothing written), untouched
sentinels beyond what each rank receives, and seeded random cases mixing all
of these.
"""
import numpy as np
import pytest
import torch

import bmm_reducescatter_alltoall_gb300 as bra
from oracle import a2av as oa
from workloads import A2AV_CONFIGS, a2av_index, a2av_inputs

pytestmark = pytest.mark.gpu

SENT_F32 = np.array([0x7FBADBAD], dtype=np.uint32).view(np.float32)[0]
SENT_I8 = np.int8(0x5A)
BOOK_SENT = -777


def _bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint8)


def _run(sc, inputs, index, dt, L=4, guard=9, in_off=0, out_off=0):
    P = sc.shape[0]
    tdt = torch.float32 if dt == "fp32" else torch.int8
    ndt = np.float32 if dt == "fp32" else np.int8
    sent = SENT_F32 if dt == "fp32" else SENT_I8
    ins = []
    for a in inputs:
        buf = torch.zeros(len(a) + in_off, dtype=tdt, device="cuda")
        v = buf[in_off:]
        v.copy_(torch.from_numpy(np.ascontiguousarray(a)))
        ins.append(v)
    idx = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in index]
    cols = np.maximum(sc, 0).sum(axis=0)
    init = [np.full(int(c) + guard, sent, dtype=ndt) for c in cols]
    outs = []
    for j in range(P):
        buf = torch.from_numpy(np.concatenate([np.full(out_off, sent, dtype=ndt), init[j]])).cuda()
        outs.append(buf[out_off:])
    scd = torch.from_numpy(np.ascontiguousarray(sc)).cuda()
    book = [torch.full((P, P), BOOK_SENT, dtype=torch.int64, device="cuda") for _ in range(3)]
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    bra.indexed_all_to_all_v(ins, idx, scd, outs, L, status=status, send_displs=book[0],
                             recv_counts=book[1], recv_displs=book[2])
    torch.cuda.synchronize()
    got = [o.cpu().numpy() for o in outs]
    return got, [b.cpu().numpy() for b in book], int(status.item()), init


def _check_against_oracle(sc, inputs, index, dt, **kw):
    got, book, st, init = _run(sc, inputs, index, dt, **kw)
    ref = oa.indexed_all_to_all_v(inputs, index, sc, init)
    for j in range(sc.shape[0]):
        np.testing.assert_array_equal(_bits(got[j]), _bits(ref["out"][j]), err_msg=f"rank {j}")
    np.testing.assert_array_equal(book[0], ref["send_displs"])
    np.testing.assert_array_equal(book[1], ref["recv_counts"])
    np.testing.assert_array_equal(book[2], ref["recv_displs"])
    assert st == (0 if ref["invalid"] == 0 else bra.ERR_INVALID)
    return ref


def _case(P, seed, dt, hi=300, extra=0):
    rng = np.random.default_rng(seed)
    sc = rng.integers(0, hi + 1, size=(P, P)).astype(np.int64)
    sc[rng.random((P, P)) < 0.25] = 0
    lens = [int(sc[i].sum()) + extra for i in range(P)]
    if dt == "fp32":
        inputs = [rng.standard_normal(n).astype(np.float32) for n in lens]
    else:
        inputs = [rng.integers(-128, 128, size=n, dtype=np.int8) for n in lens]
    return sc, inputs, lens


@pytest.mark.parametrize("dt", ["fp32", "int8"])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 32, 64])
@pytest.mark.parametrize("kind", ["identity", "perm", "random"])
def test_small_cases_bit_exact(P, dt, kind):
    extra = 17 if kind == "random" else 0
    sc, inputs, lens = _case(P, seed=P * 7 + len(kind), dt=dt, extra=extra)
    index = a2av_index(sc, lens, kind, seed=P)
    _check_against_oracle(sc, inputs, index, dt, L=max(P, 1))


@pytest.mark.parametrize("P,L", [(8, 1), (8, 3), (8, 8), (32, 64), (32, 152), (5, 1000)])
def test_launch_width_is_exactly_core_num(P, L, capfd, monkeypatch):
    """The indexed exchange launches exactly L blocks (one per SM, at most
    the SM count) and stays bit-exact at every width."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    monkeypatch.setenv("BRA_LOG", "1")
    sc, inputs, lens = _case(P, seed=900 + P + L, dt="int8", hi=4000 if P <= 8 else 400)
    index = a2av_index(sc, lens, "perm", seed=L)
    _check_against_oracle(sc, inputs, index, "int8", L=L)
    assert f"L={L} blocks={min(L, sms)}" in capfd.readouterr().err


def test_identity_index_equals_all_to_all_v():
    cfg = A2AV_CONFIGS["P8_L10_fp32_uniform4096"]
    sc, inputs = a2av_inputs(cfg)
    index = a2av_index(sc, [len(a) for a in inputs], "identity")
    got, book, st, _ = _run(sc, inputs, index, "fp32", L=cfg.L)
    ins = [torch.from_numpy(a).cuda() for a in inputs]
    outs = [torch.empty(len(g), dtype=torch.float32, device="cuda") for g in got]
    for o, g in zip(outs, got):
        o.copy_(torch.from_numpy(g))                 # same tails as the indexed run
    plain = bra.all_to_all_v(ins, torch.from_numpy(sc).cuda(), outs, cfg.L)
    torch.cuda.synchronize()
    assert st == 0
    for o, g in zip(plain["out"], got):
        np.testing.assert_array_equal(_bits(o.cpu().numpy()), _bits(g))
    np.testing.assert_array_equal(book[0], plain["send_displs"].cpu().numpy())
    np.testing.assert_array_equal(book[2], plain["recv_displs"].cpu().numpy())


@pytest.mark.parametrize("name,kind", [("P32_L64_int8_dirichlet0.3", "perm"),
                                       ("P8_L10_fp32_uniform4096", "perm"),
                                       ("P8_L10_fp32_uniform4096", "random")])
def test_full_size_workloads(name, kind):
    cfg = A2AV_CONFIGS[name]
    sc, inputs = a2av_inputs(cfg, extra=0 if kind == "perm" else 1000)
    index = a2av_index(sc, [len(a) for a in inputs], kind, seed=5)
    _check_against_oracle(sc, inputs, index, cfg.dtype, L=cfg.L, guard=64)


@pytest.mark.parametrize("in_off,out_off", [(1, 3), (3, 1), (2, 2)])
def test_unaligned_views(in_off, out_off):
    for dt in ("fp32", "int8"):
        sc, inputs, lens = _case(5, seed=in_off * 10 + out_off, dt=dt, extra=5)
        index = a2av_index(sc, lens, "random", seed=3)
        _check_against_oracle(sc, inputs, index, dt, in_off=in_off, out_off=out_off)


def test_out_of_range_index_not_delivered_and_reported():
    sc, inputs, lens = _case(4, seed=77, dt="fp32", extra=3)
    index = a2av_index(sc, lens, "random", seed=4)
    rng = np.random.default_rng(8)
    for i in range(4):
        if len(index[i]):
            bad = rng.choice(len(index[i]), size=min(5, len(index[i])), replace=False)
            index[i][bad[::2]] = -1 - rng.integers(0, 1 << 40, size=len(bad[::2]))
            index[i][bad[1::2]] = lens[i] + rng.integers(0, 1 << 40, size=len(bad[1::2]))
    ref = _check_against_oracle(sc, inputs, index, "fp32")
    assert ref["invalid"] > 0


def test_zero_counts_write_only_bookkeeping():
    P = 6
    sc = np.zeros((P, P), dtype=np.int64)
    inputs = [np.zeros(0, dtype=np.float32) for _ in range(P)]
    got, book, st, init = _run(sc, inputs, [np.zeros(0, np.int64)] * P, "fp32")
    assert st == 0
    for g, i0 in zip(got, init):
        np.testing.assert_array_equal(_bits(g), _bits(i0))
    for b in book:
        assert (b == 0).all()


def test_negative_count_rejects_the_whole_call():
    sc, inputs, lens = _case(4, seed=9, dt="int8")
    index = a2av_index(sc, lens, "perm", seed=1)
    sc[2, 1] = -3
    got, book, st, init = _run(sc, inputs, index, "int8")
    assert st == bra.ERR_INVALID
    for g, i0 in zip(got, init):
        np.testing.assert_array_equal(_bits(g), _bits(i0))
    for b in book:
        assert (b == BOOK_SENT).all()


def test_null_output_that_would_receive_rejects_the_whole_call():
    """Through the C ABI with an explicit NULL out[3]: rank 3 would receive,
    so the kernel writes nothing and reports BRA_ERR_INVALID; a NULL out[2]
    that receives nothing is fine."""
    import ctypes
    P = 4
    sc = np.array([[1, 2, 0, 1], [0, 1, 0, 2], [3, 0, 0, 1], [1, 1, 0, 0]], dtype=np.int64)
    rows = sc.sum(axis=1)
    ins = [torch.arange(int(r), dtype=torch.float32, device="cuda") for r in rows]
    idx = [torch.arange(int(r), dtype=torch.int64, device="cuda") for r in rows]
    cols = sc.sum(axis=0)
    outs = [torch.full((int(c) + 4,), -1.0, device="cuda") for c in cols]
    scd = torch.from_numpy(sc).cuda()
    book = [torch.full((P, P), BOOK_SENT, dtype=torch.int64, device="cuda") for _ in range(3)]
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    lib = bra.library()
    lens = (ctypes.c_int64 * P)(*[int(r) for r in rows])

    def call(out_ptrs):
        return lib.indexed_all_to_all_v(
            bra._ptr_array([t.data_ptr() for t in ins]), lens,
            bra._ptr_array([t.data_ptr() for t in idx]), scd.data_ptr(), book[0].data_ptr(),
            book[1].data_ptr(), book[2].data_ptr(), bra._ptr_array(out_ptrs), P, 4, bra.FP32,
            status.data_ptr(), None)

    ptrs = [t.data_ptr() for t in outs]
    assert call([ptrs[0], ptrs[1], 0, ptrs[3]]) == 0          # rank 2 receives nothing
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for b in book:
        b.fill_(BOOK_SENT)
    for o in outs:
        o.fill_(-1.0)
    assert call([ptrs[0], ptrs[1], ptrs[2], 0]) == 0          # rank 3 would receive
    torch.cuda.synchronize()
    assert int(status.item()) == bra.ERR_INVALID
    for o in outs:
        assert (o == -1.0).all().item()
    for b in book:
        assert (b == BOOK_SENT).all().item()


@pytest.mark.parametrize("k", range(16))
def test_random_indexed_exchanges_match_the_oracle(k):
    """Random rank counts, launch widths, dtypes, count mixes (zeros, a few
    large pieces among many small ones), index kinds (identity, permutation,
    repeats with unused input), a sprinkling of out-of-range index values and
    buffer offsets, bit-exact against the oracle, with the out-of-range
    elements reported and left undelivered."""
    rng = np.random.default_rng(7000 + k)
    P = int(rng.choice([1, 2, 3, 5, 8, 13, 32, 47, 64]))
    dt = "int8" if rng.random() < 0.6 else "fp32"
    L = int(rng.choice([1, 2, P, 2 * P + 1, 64, 152, 1000]))
    big = rng.integers(0, 1 << 15, size=(P, P))
    small = rng.integers(0, 40, size=(P, P))
    sc = np.where(rng.random((P, P)) < 4.0 / max(P, 4), big, small).astype(np.int64)
    sc[rng.random((P, P)) < 0.3] = 0
    kind = str(rng.choice(["identity", "perm", "random"]))
    extra = int(rng.integers(1, 200)) if kind == "random" else 0
    lens = [int(sc[i].sum()) + extra for i in range(P)]
    inputs = [(rng.integers(-128, 128, size=n, dtype=np.int8) if dt == "int8"
               else rng.standard_normal(n).astype(np.float32)) for n in lens]
    index = a2av_index(sc, lens, kind, seed=int(rng.integers(0, 1 << 30)))
    bad = 0
    if rng.random() < 0.5:
        for i in range(P):
            n = int(sc[i].sum())
            if n == 0:
                continue
            at = rng.choice(n, size=min(n, int(rng.integers(1, 6))), replace=False)
            index[i][at] = np.where(rng.random(len(at)) < 0.5,
                                    -1 - rng.integers(0, 1 << 40, size=len(at)),
                                    lens[i] + rng.integers(0, 1 << 40, size=len(at)))
            bad += len(at)
    offs = 4 if dt == "int8" else 2
    ref = _check_against_oracle(sc, inputs, index, dt, L=L, in_off=int(rng.integers(0, offs)),
                                out_off=int(rng.integers(0, offs)))
    assert ref["invalid"] == bad
    assert bra.fault_status() == 0
