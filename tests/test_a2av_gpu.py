"""all_to_all_v on the GPU against the CPU oracle: bit-exact.

Covers the two workloads (fp32 P=8 L=10 uniform counts; int8 P=32 L=64
Dirichlet-skewed counts), the count-matrix categories of the PyPTO system
test (0 / 1 / capacity / over capacity / negative), all-to-self, P from 1 to
64, launch widths below, at and above P, source and destination buffers at
every byte misalignment, and untouched sentinels beyond what each rank
receives.
"""
import itertools

import numpy as np
import pytest
import torch

import bmm_reducescatter_alltoall_gb300 as bra
from oracle import a2av as oa
from workloads import A2AV_CONFIGS, a2av_inputs

pytestmark = pytest.mark.gpu

SENT_F32 = np.array([0x7FBADBAD], dtype=np.uint32).view(np.float32)[0]
SENT_I8 = np.int8(0x5A)
BOOK_SENT = -777


def _np_dtype(dt):
    return np.float32 if dt == "fp32" else np.int8


def _torch_dtype(dt):
    return torch.float32 if dt == "fp32" else torch.int8


def _bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint8)


def run_case(sc, inputs, dt, L, in_off=None, out_off=None, guard=37, checked=False,
             capacity=None):
    """Run the GPU exchange and the oracle; return both plus the raw buffers."""
    P = sc.shape[0]
    tdt, ndt = _torch_dtype(dt), _np_dtype(dt)
    sent = SENT_F32 if dt == "fp32" else SENT_I8
    in_off = in_off or [0] * P
    out_off = out_off or [0] * P
    cols = np.maximum(sc, 0).sum(axis=0)
    cap = [int(c) + guard for c in cols] if capacity is None else list(capacity)
    ins, in_bufs = [], []
    for i in range(P):
        buf = torch.zeros(len(inputs[i]) + in_off[i], dtype=tdt, device="cuda")
        v = buf[in_off[i]:]
        v.copy_(torch.from_numpy(np.ascontiguousarray(inputs[i])))
        ins.append(v)
        in_bufs.append(buf)
    outs, out_bufs = [], []
    for j in range(P):
        host = np.full(cap[j] + out_off[j], sent, dtype=ndt)
        buf = torch.from_numpy(host).cuda()
        outs.append(buf[out_off[j]:])
        out_bufs.append(buf)
    sc_d = torch.from_numpy(np.ascontiguousarray(sc)).cuda()
    book = [torch.full((P, P), BOOK_SENT, dtype=torch.int64, device="cuda") for _ in range(3)]
    if checked:
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        bra.all_to_all_v_checked(ins, sc_d, outs, L, out_capacity=cap, status=status,
                                 send_displs=book[0], recv_counts=book[1], recv_displs=book[2])
    else:
        status = None
        bra.all_to_all_v(ins, sc_d, outs, L, send_displs=book[0], recv_counts=book[1],
                         recv_displs=book[2])
    torch.cuda.synchronize()
    got = {
        "out": [b.cpu().numpy() for b in out_bufs],
        "book": [b.cpu().numpy() for b in book],
        "status": None if status is None else int(status.item()),
        "sc_after": sc_d.cpu().numpy(),
        "in_after": [b.cpu().numpy() for b in in_bufs],
    }
    return got, cap, out_off


def check_exact(sc, inputs, dt, L, **kw):
    got, cap, out_off = run_case(sc, inputs, dt, L, **kw)
    P = sc.shape[0]
    ndt = _np_dtype(dt)
    sent = SENT_F32 if dt == "fp32" else SENT_I8
    init = [np.full(cap[j], sent, dtype=ndt) for j in range(P)]
    ref = oa.all_to_all_v([np.asarray(a, dtype=ndt) for a in inputs], sc, init)
    for j in range(P):
        buf = got["out"][j]
        assert (_bits(buf[:out_off[j]]) == _bits(np.full(out_off[j], sent, dtype=ndt))).all()
        np.testing.assert_array_equal(_bits(buf[out_off[j]:]), _bits(ref["out"][j]),
                                      err_msg=f"rank {j}")
    np.testing.assert_array_equal(got["book"][0], ref["send_displs"])
    np.testing.assert_array_equal(got["book"][1], ref["recv_counts"])
    np.testing.assert_array_equal(got["book"][2], ref["recv_displs"])
    np.testing.assert_array_equal(got["sc_after"], sc)
    return got


def _random_case(P, dt, seed, hi=300, zero_frac=0.25):
    rng = np.random.default_rng(seed)
    sc = rng.integers(0, hi + 1, size=(P, P)).astype(np.int64)
    sc[rng.random((P, P)) < zero_frac] = 0
    ndt = _np_dtype(dt)
    if dt == "fp32":
        inputs = [rng.standard_normal(int(sc[i].sum())).astype(ndt) for i in range(P)]
    else:
        inputs = [rng.integers(-128, 128, size=int(sc[i].sum()), dtype=np.int8) for i in range(P)]
    return sc, inputs


@pytest.mark.parametrize("name", list(A2AV_CONFIGS))
def test_workloads_bit_exact(name):
    cfg = A2AV_CONFIGS[name]
    sc, inputs = a2av_inputs(cfg)
    assert bra.cal_all_to_all_v_blocks(cfg.P, cfg.L) == oa.cal_all_to_all_v_blocks(cfg.P, cfg.L)
    got = check_exact(sc, inputs, cfg.dtype, cfg.L)
    assert bra.fault_status() == 0
    del got


@pytest.mark.parametrize("name,field,value", [
    ("P32_L64_int8_dirichlet0.3", "scale", 1 << 23),     # ~8 MiB sent per rank
    ("P8_L10_fp32_uniform4096", "count_max", 1 << 20),   # ~2 MiB per pair
])
def test_large_sizes_bit_exact(name, field, value):
    """Sizes from the upper part of the bench's size sweep (256 MiB moved)."""
    cfg = A2AV_CONFIGS[name].replace(**{field: value})
    sc, inputs = a2av_inputs(cfg)
    check_exact(sc, inputs, cfg.dtype, cfg.L, guard=5)
    assert bra.fault_status() == 0


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 32, 64])
@pytest.mark.parametrize("dt", ["fp32", "int8"])
def test_rank_counts_and_launch_widths(P, dt):
    widths = sorted({1, 3, max(1, P - 1), P, P + 1, 2 * P + 3, 64})
    for k, L in enumerate(widths):
        sc, inputs = _random_case(P, dt, seed=1000 * P + k, hi=200 if P <= 8 else 40)
        check_exact(sc, inputs, dt, L)


@pytest.mark.parametrize("P,L", [(8, 1), (8, 3), (8, 8), (8, 19), (32, 64), (32, 10**6),
                                 (64, 200), (3, 2)])
def test_launch_blocks_follow_core_num(P, L, capfd, monkeypatch):
    """The exchange launches B = CalAllToAllVBlocks(P, L) blocks, one per SM,
    at most the SM count, and stays bit-exact at every width."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B = bra.cal_all_to_all_v_blocks(P, L)
    want = min(B, sms)
    assert bra.all_to_all_v_launch_blocks(P, L) == want
    monkeypatch.setenv("BRA_LOG", "1")
    sc, inputs = _random_case(P, "int8", seed=7 * P + L % 1009, hi=5000 if P <= 8 else 600)
    check_exact(sc, inputs, "int8", L, in_off=[k % 16 for k in range(P)])
    assert f"B={B} blocks={want}" in capfd.readouterr().err


@pytest.mark.parametrize("L", [1, 5, 64, 152])
def test_sixty_four_ranks_many_chunks(L):
    """P = 64 (the largest count matrix, the shortest ring) with pieces that
    span many ring wraps per block, from one block up to one per SM."""
    sc, inputs = _random_case(64, "int8", seed=640 + L, hi=12000, zero_frac=0.3)
    check_exact(sc, inputs, "int8", L, in_off=[(3 * k) % 16 for k in range(64)])


@pytest.mark.parametrize("dt", ["fp32", "int8"])
def test_every_byte_misalignment(dt):
    P = 4
    es = 4 if dt == "fp32" else 1
    offs = list(range(0, 16 // es))
    for k, (io, oo) in enumerate(itertools.product(offs, offs)):
        sc, inputs = _random_case(P, dt, seed=77 + k, hi=97)
        check_exact(sc, inputs, dt, 5, in_off=[io, (io + 1) % len(offs), io, 0],
                    out_off=[oo, 0, (oo + 3) % len(offs), oo])


@pytest.mark.parametrize("dt", ["fp32", "int8"])
def test_count_categories(dt):
    P = 4
    ndt = _np_dtype(dt)
    rng = np.random.default_rng(5)
    mk = lambda sc: [rng.integers(-100, 100, size=int(max(0, sc[i].sum()))).astype(ndt)
                     for i in range(P)]
    zeros = np.zeros((P, P), dtype=np.int64)
    ones = np.ones((P, P), dtype=np.int64)
    self_only = np.diag(np.array([5, 0, 17, 1], dtype=np.int64))
    for sc in (zeros, ones, self_only):
        check_exact(sc, mk(sc), dt, P)
        got = check_exact(sc, mk(sc), dt, P, checked=True)
        assert got["status"] == 0


def test_big_single_pair():
    sc = np.array([[0, 3_000_001], [5, 0]], dtype=np.int64)
    rng = np.random.default_rng(9)
    inputs = [rng.integers(-128, 128, size=int(sc[i].sum()), dtype=np.int8) for i in range(2)]
    check_exact(sc, inputs, "int8", 64, in_off=[3, 0], out_off=[0, 11])


@pytest.mark.parametrize("dt", ["fp32", "int8"])
def test_capacity_exact_and_over(dt):
    P = 3
    sc, inputs = _random_case(P, dt, seed=11, hi=50, zero_frac=0.0)
    cols = sc.sum(axis=0)
    got = check_exact(sc, inputs, dt, 4, checked=True, capacity=[int(c) for c in cols])
    assert got["status"] == 0
    cap = [int(c) for c in cols]
    cap[1] -= 1                                   # one element short at rank 1
    got, _, _ = run_case(sc, inputs, dt, 4, checked=True, capacity=cap)
    assert got["status"] == bra.ERR_INVALID
    _assert_nothing_written(got, dt)


def _assert_nothing_written(got, dt):
    sent = SENT_F32 if dt == "fp32" else SENT_I8
    ndt = _np_dtype(dt)
    for buf in got["out"]:
        assert (_bits(buf) == _bits(np.full(len(buf), sent, dtype=ndt))).all()
    for b in got["book"]:
        assert (b == BOOK_SENT).all()


@pytest.mark.parametrize("dt", ["fp32", "int8"])
@pytest.mark.parametrize("checked", [False, True])
def test_negative_count_writes_nothing(dt, checked):
    P = 4
    sc, inputs = _random_case(P, dt, seed=12, hi=30, zero_frac=0.0)
    sc[2, 1] = -1
    inputs = [a[:max(0, int(sc[i].sum()))] for i, a in enumerate(inputs)]
    got, _, _ = run_case(sc, inputs, dt, 4, checked=checked, guard=64)
    if checked:
        assert got["status"] == bra.ERR_INVALID
    _assert_nothing_written(got, dt)


def test_transposed_counts_invert_on_gpu():
    P = 8
    sc, inputs = _random_case(P, "fp32", seed=21, hi=500)
    tin = [torch.from_numpy(a).cuda() for a in inputs]
    cols = sc.sum(axis=0)
    mid = [torch.empty(int(c), dtype=torch.float32, device="cuda") for c in cols]
    bra.all_to_all_v(tin, torch.from_numpy(sc).cuda(), mid, 10)
    back = [torch.empty(len(a), dtype=torch.float32, device="cuda") for a in inputs]
    bra.all_to_all_v(mid, torch.from_numpy(sc.T.copy()).cuda(), back, 10)
    torch.cuda.synchronize()
    for a, b in zip(inputs, back):
        np.testing.assert_array_equal(a.view(np.uint32), b.cpu().numpy().view(np.uint32))


def test_repeat_calls_are_identical():
    cfg = A2AV_CONFIGS["P8_L10_fp32_uniform4096"]
    sc, inputs = a2av_inputs(cfg)
    a = check_exact(sc, inputs, "fp32", cfg.L)
    b = check_exact(sc, inputs, "fp32", cfg.L)
    for x, y in zip(a["out"], b["out"]):
        np.testing.assert_array_equal(x.view(np.uint32), y.view(np.uint32))


def test_l2_flush_reads_without_writing():
    buf = torch.arange((1 << 22) + 7, dtype=torch.int32, device="cuda").to(torch.int8)
    before = buf.clone()
    bra.l2_flush(buf)
    torch.cuda.synchronize()
    assert torch.equal(buf, before)
    with pytest.raises(bra.BraError):
        bra.l2_flush(buf[1:])                         # not 16-byte aligned


@pytest.mark.parametrize("L", [64, 1])
def test_piece_beyond_two_gib(L):
    """One pair carries 2^31 + 4099 int8 elements (element offsets and byte
    counts past 32 bits) from an input that starts 3 bytes past 16-byte
    alignment: every byte arrives, checked on the device against the input
    (the exchange's definition, out[1][n] = in[0][n]), and the bookkeeping
    matches the oracle's."""
    n = (1 << 31) + 4099
    sc = np.array([[0, n], [5, 0]], dtype=np.int64)
    g = torch.Generator(device="cuda")
    g.manual_seed(31)
    buf0 = torch.randint(-128, 128, (n + 3,), generator=g, dtype=torch.int8, device="cuda")
    in0 = buf0[3:]
    in1 = torch.tensor([1, 2, 3, 4, 5], dtype=torch.int8, device="cuda")
    out1 = torch.empty(n + 7, dtype=torch.int8, device="cuda")
    out1[n:] = 0x5A
    out0 = torch.full((5,), 0x11, dtype=torch.int8, device="cuda")
    res = bra.all_to_all_v([in0, in1], torch.from_numpy(sc).cuda(), [out0, out1], L)
    torch.cuda.synchronize()
    assert torch.equal(out1[:n], in0)
    assert (out1[n:] == 0x5A).all()
    assert torch.equal(out0, in1)
    for key, want in zip(("send_displs", "recv_counts", "recv_displs"), oa.a2av_bookkeeping(sc)):
        np.testing.assert_array_equal(res[key].cpu().numpy(), want)
    assert bra.fault_status() == 0
    del buf0, out1
    torch.cuda.empty_cache()


@pytest.mark.parametrize("k", range(24))
def test_random_exchanges_match_the_oracle(k):
    """Random rank counts, launch widths, dtypes, count mixes (zeros, a few
    large pieces among many small ones, rows of one destination) and buffer
    offsets, bit-exact against the oracle."""
    rng = np.random.default_rng(5000 + k)
    P = int(rng.choice([1, 2, 3, 5, 8, 13, 32, 47, 64]))
    dt = "int8" if rng.random() < 0.6 else "fp32"
    es = 1 if dt == "int8" else 4
    L = int(rng.choice([1, 2, P, 2 * P + 1, 64, 152, 1000]))
    big = rng.integers(0, (1 << 18) // es, size=(P, P))
    small = rng.integers(0, 40, size=(P, P))
    sc = np.where(rng.random((P, P)) < 4.0 / max(P, 4), big, small).astype(np.int64)
    sc[rng.random((P, P)) < 0.3] = 0
    if rng.random() < 0.3:                         # one row sends everything to one rank
        r = int(rng.integers(0, P))
        sc[r] = 0
        sc[r, int(rng.integers(0, P))] = int(rng.integers(1, (1 << 20) // es))
    ndt = np.int8 if dt == "int8" else np.float32
    inputs = [(rng.integers(-128, 128, size=int(sc[i].sum()), dtype=np.int8) if dt == "int8"
               else rng.standard_normal(int(sc[i].sum())).astype(np.float32)) for i in range(P)]
    offs = 16 // es
    check_exact(sc, inputs, dt, L, in_off=[int(rng.integers(0, offs)) for _ in range(P)],
                out_off=[int(rng.integers(0, offs)) for _ in range(P)])
    assert bra.fault_status() == 0
