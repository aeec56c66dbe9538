"""Host-side tests of the C ABI (no GPU needed, no kernel launched).

The library is loaded through ctypes; every symbol the public header declares
must be exported.  Pure host functions (launch width, shape inference) are
compared bit-exactly with the oracle; argument validation is driven with
stand-in pointer values on calls that must be rejected before any launch,
and with `bmm_rs_a2a_variant`, which runs the same validation without
launching, for calls that would be accepted.
"""
import ctypes
import pathlib
import itertools
import os
import re

import numpy as np
import pytest

import bmm_reducescatter_alltoall_gb300 as bra
from oracle import a2av as oa
from oracle import fused as of

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bmm_rs_a2a.h")

OK, NULLPTR, INVALID, UNSUPPORTED = 0, 161001, 161002, 161003


@pytest.fixture(scope="module")
def lib():
    return bra.library()


def _declared_functions():
    src = pathlib.Path(HEADER).read_text()
    return re.findall(r"^BRA_API\s+[\w\s\*]+?\b(\w+)\s*\(", src, flags=re.M)


def test_header_declares_the_entry_points():
    names = set(_declared_functions())
    assert {"bmm_rs_a2a", "all_to_all_v", "all_to_all_v_checked", "cal_all_to_all_v_blocks",
            "bmm_rs_a2a_infer_shape", "bra_status_str"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert bra.status_str(OK) == "BRA_OK"
    assert bra.status_str(INVALID) == "BRA_ERR_INVALID"
    assert bra.status_str(12345) == "BRA_UNKNOWN_STATUS"
    assert bra.version().count(".") == 2


def test_cal_blocks_matches_oracle(lib):
    for P in list(range(1, 40)) + [64, 1000]:
        for L in list(range(0, 130)) + [2**31 - 1, 2**31, -5]:
            assert bra.cal_all_to_all_v_blocks(P, L) == oa.cal_all_to_all_v_blocks(P, L), (P, L)
    assert bra.cal_all_to_all_v_blocks(0, 4) == -1


def test_launch_blocks_rejects_what_the_exchange_rejects(lib):
    """all_to_all_v_launch_blocks refuses the arguments all_to_all_v refuses
    (without a device, valid arguments fail only at the device query)."""
    import torch
    for P, L, code in ((0, 4, INVALID), (8, 0, INVALID), (8, 2**31, INVALID),
                       (65, 65, bra.ERR_UNSUPPORTED), (64, 2**31 - 1, INVALID)):
        with pytest.raises(bra.BraError) as e:
            bra.all_to_all_v_launch_blocks(P, L)
        assert e.value.code == code, (P, L)
    if not torch.cuda.is_available():
        with pytest.raises(bra.BraError) as e:
            bra.all_to_all_v_launch_blocks(8, 10)
        assert e.value.code == bra.ERR_CUDA


def test_infer_shape_matches_oracle_and_rules(lib):
    rng = np.random.default_rng(0)
    seen_ok = seen_bad = 0
    for _ in range(3000):
        # mostly valid draws, each perturbed in one field a third of the time
        ep = int(rng.choice([1, 2, 4, 8, 16, 32]))
        tp = int(rng.choice([1, 2, 4, 8, 16, 32]))
        E = ep * int(rng.integers(1, 34))
        t = int(rng.integers(0, 2))
        C = tp * int(rng.integers(1, 20)) + (int(rng.integers(0, tp)) if t == 0 else 0)
        M = tp * int(rng.integers(1, 3000))
        H = tp * int(rng.integers(1, 3000)) + (int(rng.integers(0, tp)) if t == 1 else 0)
        if rng.random() < 0.33:
            k = int(rng.integers(0, 7))
            if k == 0:
                ep = int(rng.choice([0, 3, 64]))
            elif k == 1:
                tp = int(rng.choice([0, 5, 64]))
            elif k == 2:
                E = int(rng.choice([0, 1, 513, E + 1]))
            elif k == 3:
                C = int(rng.choice([0, -1, C + 1]))
            elif k == 4:
                M = int(rng.choice([0, M + 1, 65536 * tp]))
            elif k == 5:
                H = int(rng.choice([0, 65536, H + 1]))
            else:
                t = int(rng.choice([-1, 2]))
        try:
            want = of.infer_shapes(ep, tp, E, C, M, H, t)
        except of.OracleParamError:
            want = None
        arrs = [(ctypes.c_int64 * 3)() for _ in range(4)]
        rc = lib.bmm_rs_a2a_infer_shape(ep, tp, E, C, M, H, t, *arrs)
        if want is None:
            assert rc == INVALID, (ep, tp, E, C, M, H, t)
            seen_bad += 1
        else:
            assert rc == OK
            got = dict(zip(("x", "w", "bias", "y"), (tuple(a) for a in arrs)))
            assert got == want
            seen_ok += 1
    assert seen_ok > 50 and seen_bad > 50
    for ep, tp, t in itertools.product((1, 2, 4, 8, 16, 32), (1, 2, 4, 8, 16, 32), (0, 1)):
        E, C, M, H = 2 * ep, 4 * tp, 6 * tp, 8 * tp
        assert bra.bmm_rs_a2a_infer_shape(ep, tp, E, C, M, H, t) == of.infer_shapes(
            ep, tp, E, C, M, H, t)


# --------------------------------------------------------------------------
# Fused-op validation
# --------------------------------------------------------------------------

class Fake:
    """Stand-in device addresses laid out like real, disjoint buffers."""

    def __init__(self, ep, tp, E, C, M, H, t, bias=True, base=1 << 40):
        sh = of.infer_shapes(ep, tp, E, C, M, H, t)
        P = ep * tp
        nbytes = lambda s, es=2: int(np.prod(s)) * es
        addr = base
        self.x, self.w, self.b, self.y = [], [], [], []
        for _ in range(P):
            for lst, n in ((self.x, nbytes(sh["x"])), (self.w, nbytes(sh["w"])),
                           (self.b, nbytes(sh["bias"], 4)), (self.y, nbytes(sh["y"]))):
                lst.append(addr)
                addr += (n + 4095) // 4096 * 4096 + 4096
        if not bias:
            self.b = None
        self.args = (ep, tp, E, C, M, H, t)

    def arrays(self):
        mk = lambda v: None if v is None else bra._ptr_array(v)
        return mk(self.x), mk(self.w), mk(self.b), mk(self.y)


def _variant(lib, f, dtype=bra.FP16, opts=None, **over):
    x, w, b, y = f.arrays()
    ep, tp, E, C, M, H, t = f.args
    p = dict(ep=ep, tp=tp, E=E, C=C, M=M, H=H, t=t)
    p.update(over)
    return lib.bmm_rs_a2a_variant(x, w, b, p["ep"], p["tp"], p["E"], p["C"], p["M"], p["H"],
                                  p["t"], dtype, y, None if opts is None else ctypes.byref(opts))


def _call_rejected(lib, f, dtype=bra.FP16, **over):
    """Call the real entry point; the arguments must be rejected."""
    x, w, b, y = f.arrays()
    ep, tp, E, C, M, H, t = f.args
    p = dict(ep=ep, tp=tp, E=E, C=C, M=M, H=H, t=t, x=x, w=w, b=b, y=y)
    p.update(over)
    assert _variant(lib, f, dtype, **{k: v for k, v in over.items() if k in "ep tp E C M H t"}) < 0 \
        or any(k in over for k in ("x", "w", "y", "b"))
    return lib.bmm_rs_a2a(p["x"], p["w"], p["b"], p["ep"], p["tp"], p["E"], p["C"], p["M"],
                          p["H"], p["t"], dtype, p["y"], None)


def test_valid_shapes_choose_a_variant(lib):
    f = Fake(4, 2, 16, 12, 12, 4, 1)                  # M/tp = 6: not 16-byte rows
    assert _variant(lib, f) == bra.VARIANT_TCR        # tensor cores fed by row-class TMA maps
    g = Fake(8, 4, 64, 512, 8192, 4096, 1)
    assert _variant(lib, g) == bra.VARIANT_TC2
    assert _variant(lib, Fake(8, 2, 64, 256, 4096, 4096, 0), bra.BF16) == bra.VARIANT_TC2
    assert _variant(lib, Fake(2, 2, 4, 96, 256, 512, 0)) == bra.VARIANT_TC     # 4 pair tiles
    # decode-like token counts: <= 128 rows per group stream weights on one-CTA tiles
    assert _variant(lib, Fake(8, 4, 64, 16, 8192, 4096, 1)) == bra.VARIANT_TC
    assert _variant(lib, Fake(8, 4, 64, 32, 8192, 4096, 1)) == bra.VARIANT_TC2
    assert _variant(lib, Fake(2, 2, 4, 4, 16, 20, 0)) == bra.VARIANT_TCR    # H/tp = 10
    # odd M/tp and H: 8 row classes each; 16 maps a rank fit one TP group of 8
    # ranks in a launch (176 maps), not one of 16: operands staged by loads
    assert _variant(lib, Fake(2, 8, 4, 16, 8 * 3, 5, 1)) == bra.VARIANT_TCR
    assert _variant(lib, Fake(2, 16, 4, 16, 16 * 3, 5, 1)) == bra.VARIANT_TCU
    # an operand that is not even element-aligned: only the generic kernel
    odd = Fake(4, 2, 16, 12, 12, 4, 1)
    odd.x[3] += 1
    assert _variant(lib, odd) == bra.VARIANT_SIMT


def test_forced_variant(lib, monkeypatch):
    monkeypatch.setenv("BRA_FORCE_VARIANT", "tc2")
    assert _variant(lib, Fake(8, 4, 64, 512, 8192, 4096, 1)) == bra.VARIANT_TC2
    assert _variant(lib, Fake(4, 2, 16, 12, 12, 4, 1)) == -UNSUPPORTED
    monkeypatch.setenv("BRA_FORCE_VARIANT", "simt")
    assert _variant(lib, Fake(8, 4, 64, 512, 8192, 4096, 1)) == bra.VARIANT_SIMT
    monkeypatch.setenv("BRA_FORCE_VARIANT", "tc")
    assert _variant(lib, Fake(4, 2, 16, 12, 12, 4, 1)) == -UNSUPPORTED
    monkeypatch.setenv("BRA_FORCE_VARIANT", "tcu")
    assert _variant(lib, Fake(8, 4, 64, 512, 8192, 4096, 1)) == bra.VARIANT_TCU
    assert _variant(lib, Fake(4, 2, 16, 12, 12, 4, 1)) == bra.VARIANT_TCU
    odd = Fake(4, 2, 16, 12, 12, 4, 1)
    odd.w[0] += 1
    assert _variant(lib, odd) == -UNSUPPORTED
    monkeypatch.setenv("BRA_FORCE_VARIANT", "tcr")
    assert _variant(lib, Fake(8, 4, 64, 512, 8192, 4096, 1)) == bra.VARIANT_TCR
    assert _variant(lib, Fake(4, 2, 16, 12, 12, 4, 1)) == bra.VARIANT_TCR
    assert _variant(lib, odd) == -UNSUPPORTED
    assert _variant(lib, Fake(2, 16, 4, 16, 16 * 3, 5, 1)) == -UNSUPPORTED


@pytest.mark.parametrize("over", [
    dict(ep=3), dict(tp=64), dict(ep=0), dict(t=2), dict(t=-1), dict(E=1), dict(E=514),
    dict(E=12, ep=8), dict(E=264, ep=8), dict(H=0), dict(H=65536), dict(M=7, tp=2),
    dict(M=2 * 65536, tp=1), dict(C=0), dict(C=-3)])
def test_attribute_rules_invalid(lib, over):
    f = Fake(2, 2, 8, 4, 8, 8, 0)
    assert _variant(lib, f, **over) == -INVALID
    assert _call_rejected(lib, f, **over) == INVALID


def test_shape_divisibility_per_shard_type(lib):
    assert _variant(lib, Fake(2, 2, 8, 4, 8, 8, 0), H=9) == -INVALID       # H % tp, type 0
    assert _variant(lib, Fake(2, 2, 8, 4, 8, 8, 1), C=5) == -INVALID       # C % tp, type 1
    assert _variant(lib, Fake(2, 2, 8, 4, 8, 8, 1), H=9) > 0               # fine for type 1
    assert _variant(lib, Fake(2, 2, 8, 4, 8, 8, 0), C=5) > 0               # fine for type 0


def test_dtype_rule(lib):
    f = Fake(2, 2, 8, 4, 8, 8, 0)
    for dt in (bra.FP32, bra.INT8, 7, -1):
        assert _variant(lib, f, dt) == -INVALID
        assert _call_rejected(lib, f, dt, ep=3) == INVALID


def test_null_pointers(lib):
    f = Fake(2, 2, 8, 4, 8, 8, 0)
    assert _call_rejected(lib, f, x=None) == NULLPTR
    assert _call_rejected(lib, f, w=None) == NULLPTR
    assert _call_rejected(lib, f, y=None) == NULLPTR
    for field in ("x", "w", "y"):
        g = Fake(2, 2, 8, 4, 8, 8, 0)
        getattr(g, field)[3] = 0
        assert _variant(lib, g) == -NULLPTR
        x, w, b, y = g.arrays()
        assert lib.bmm_rs_a2a(x, w, b, 2, 2, 8, 4, 8, 8, 0, bra.FP16, y, None) == NULLPTR


def test_bias_all_or_nothing(lib):
    g = Fake(2, 2, 8, 4, 8, 8, 0)
    g.b[1] = 0
    assert _variant(lib, g) == -INVALID
    x, w, b, y = g.arrays()
    assert lib.bmm_rs_a2a(x, w, b, 2, 2, 8, 4, 8, 8, 0, bra.FP16, y, None) == INVALID
    h = Fake(2, 2, 8, 4, 8, 8, 0)
    h.b = [0, 0, 0, 0]
    assert _variant(lib, h) > 0                   # all-null bias = no bias


def test_aliasing_rules(lib):
    g = Fake(2, 2, 8, 4, 8, 8, 0)
    g.y[2] = g.x[1]                               # output == input
    assert _variant(lib, g) == -INVALID
    g = Fake(2, 2, 8, 4, 8, 8, 0)
    g.y[0] = g.y[3]                               # two outputs share memory
    assert _variant(lib, g) == -INVALID
    g = Fake(2, 2, 8, 4, 8, 8, 0)
    g.y[1] = g.w[2] + 64                          # output overlaps the inside of a weight
    assert _variant(lib, g) == -INVALID
    g = Fake(2, 2, 8, 4, 8, 8, 0)
    g.w[1] = g.w[0]                               # shared weights are fine (read only)
    assert _variant(lib, g) > 0
    x, w, b, y = Fake(2, 2, 8, 4, 8, 8, 0).arrays()
    g = Fake(2, 2, 8, 4, 8, 8, 0)
    g.y[3] = g.b[0]
    x, w, b, y = g.arrays()
    assert lib.bmm_rs_a2a(x, w, b, 2, 2, 8, 4, 8, 8, 0, bra.FP16, y, None) == INVALID


def test_options_select_the_variant_and_are_checked(lib, monkeypatch):
    monkeypatch.delenv("BRA_FORCE_VARIANT", raising=False)
    g = Fake(8, 4, 64, 512, 8192, 4096, 1)
    assert _variant(lib, g, opts=bra._options(False, "tc")) == bra.VARIANT_TC
    assert _variant(lib, g, opts=bra._options(True, "simt")) == bra.VARIANT_SIMT
    monkeypatch.setenv("BRA_FORCE_VARIANT", "simt")           # options win over the env
    assert _variant(lib, g, opts=bra._options(False, "tc2")) == bra.VARIANT_TC2
    bad = bra._options(False, None)
    bad.variant = 9
    assert _variant(lib, g, opts=bad) == -INVALID
    bad = bra._options(False, None)
    bad.x_pitch = -8
    assert _variant(lib, g, opts=bad) == -INVALID
    x, w, b, y = g.arrays()
    assert lib.bmm_rs_a2a_ex(x, w, b, 8, 4, 64, 512, 8192, 4096, 1, bra.FP16, y,
                             ctypes.byref(bad), None) == INVALID
    with pytest.raises(ValueError):
        bra._options(False, "fastest")


def test_tc_alignment_predicate(lib):
    # output rows or pointers without 16-byte alignment keep the TMA kernels
    # (their epilogue stores element by element): H/tp = 12, odd y offsets
    h = Fake(2, 2, 4, 64, 256, 24, 0)
    assert _variant(lib, h) == bra.VARIANT_TC
    h.y[1] += 2
    assert _variant(lib, h) == bra.VARIANT_TC
    h.y[1] += 1                                   # not even element-aligned
    assert _variant(lib, h) == bra.VARIANT_SIMT
    g = Fake(2, 2, 8, 128, 128, 256, 0)
    assert _variant(lib, g) in (bra.VARIANT_TC, bra.VARIANT_TC2)
    g.x[1] += 2                                   # 2-byte aligned only: row-class TMA
    assert _variant(lib, g) == bra.VARIANT_TCR
    g.x[1] += 1                                   # not even element-aligned
    assert _variant(lib, g) == bra.VARIANT_SIMT


# --------------------------------------------------------------------------
# all_to_all_v validation
# --------------------------------------------------------------------------

def _a2av(lib, P=4, L=4, dtype=bra.FP32, ins=None, outs=None, sc=1 << 30, sd=2 << 30,
          rc=3 << 30, rd=4 << 30, checked=False, cap=None, status=5 << 30):
    ins = [(10 + k) << 32 for k in range(P)] if ins is None else ins
    outs = [(100 + k) << 32 for k in range(P)] if outs is None else outs
    ip = bra._ptr_array(ins) if ins != "null" else None
    op = bra._ptr_array(outs) if outs != "null" else None
    if not checked:
        return lib.all_to_all_v(ip, sc, sd, rc, rd, op, P, L, dtype, None)
    capp = None if cap == "null" else (ctypes.c_int64 * max(P, 1))(*([1 << 20] * max(P, 1)))
    return lib.all_to_all_v_checked(ip, sc, sd, rc, rd, op, P, L, dtype, capp, status, None)


@pytest.mark.parametrize("checked", [False, True])
def test_a2av_rejections(lib, checked):
    kw = dict(checked=checked)
    assert _a2av(lib, P=0, **kw) == INVALID
    assert _a2av(lib, P=-1, **kw) == INVALID
    assert _a2av(lib, L=0, **kw) == INVALID
    assert _a2av(lib, L=2**31, **kw) == INVALID
    for dt in (bra.FP16, bra.BF16, 9):
        assert _a2av(lib, dtype=dt, **kw) == INVALID
    assert _a2av(lib, ins="null", **kw) == NULLPTR
    assert _a2av(lib, outs="null", **kw) == NULLPTR
    for key in ("sc", "sd", "rc", "rd"):
        assert _a2av(lib, **{key: None}, **kw) == NULLPTR
    # a NULL entry is fine on the host (a rank may have nothing to move)
    assert _a2av(lib, ins=[1 << 32, 0, 3 << 32, 4 << 32], outs=[0, 0, 0, 0], P=4,
                 dtype=9, **kw) == INVALID
    ins = [(10 + k) << 32 for k in range(4)]
    assert _a2av(lib, ins=ins, outs=[5 << 40, ins[2], 6 << 40, 7 << 40], **kw) == INVALID
    assert _a2av(lib, outs=[5 << 40, 6 << 40, 5 << 40, 7 << 40], **kw) == INVALID
    assert _a2av(lib, P=65, L=65, **kw) == UNSUPPORTED
    # B * P must fit a 32-bit grid: P = 64 with L near INT32_MAX
    assert _a2av(lib, P=64, L=2**31 - 1, **kw) == INVALID
    if checked:
        assert _a2av(lib, cap="null", **kw) == NULLPTR
        assert _a2av(lib, status=None, **kw) == NULLPTR


def _ia2av(lib, P=4, L=4, dtype=bra.INT8, ins=None, lens=None, idx=None, outs=None,
           sc=1 << 30, sd=2 << 30, rc=3 << 30, rd=4 << 30, status=None):
    ins = [(10 + k) << 32 for k in range(P)] if ins is None else ins
    idx = [(20 + k) << 32 for k in range(P)] if idx is None else idx
    outs = [(100 + k) << 32 for k in range(P)] if outs is None else outs
    lens = [16] * max(P, 1) if lens is None else lens
    ip = bra._ptr_array(ins) if ins != "null" else None
    xp = bra._ptr_array(idx) if idx != "null" else None
    op = bra._ptr_array(outs) if outs != "null" else None
    lp = (ctypes.c_int64 * len(lens))(*lens) if lens != "null" else None
    return lib.indexed_all_to_all_v(ip, lp, xp, sc, sd, rc, rd, op, P, L, dtype, status, None)


def test_indexed_a2av_rejections(lib):
    """Every rejection of the indexed exchange happens on the host, before any
    launch."""
    assert _ia2av(lib, P=0) == INVALID
    assert _ia2av(lib, L=0) == INVALID
    assert _ia2av(lib, L=2**31) == INVALID
    for dt in (bra.FP16, bra.BF16, 9):
        assert _ia2av(lib, dtype=dt) == INVALID
    for key in ("ins", "idx", "outs", "lens"):
        assert _ia2av(lib, **{key: "null"}) == NULLPTR
    for key in ("sc", "sd", "rc", "rd"):
        assert _ia2av(lib, **{key: None}) == NULLPTR
    assert _ia2av(lib, lens=[16, -1, 16, 16]) == INVALID
    assert _ia2av(lib, ins=[1 << 32, 0, 3 << 32, 4 << 32]) == NULLPTR   # in_len 16, NULL input
    ins = [(10 + k) << 32 for k in range(4)]
    idx = [(20 + k) << 32 for k in range(4)]
    assert _ia2av(lib, outs=[5 << 40, ins[2], 6 << 40, 7 << 40]) == INVALID
    assert _ia2av(lib, outs=[5 << 40, 6 << 40, idx[3], 7 << 40]) == INVALID
    assert _ia2av(lib, outs=[5 << 40, 6 << 40, 5 << 40, 7 << 40]) == INVALID
    assert _ia2av(lib, P=65, L=65, lens=[1] * 65) == UNSUPPORTED
    assert _ia2av(lib, P=64, L=2**31 - 1, lens=[1] * 64) == INVALID
    # a NULL input is fine when it holds no element: the call gets as far as
    # the aliasing rule
    assert _ia2av(lib, ins=[0] * 4, lens=[0] * 4,
                  outs=[5 << 40, 6 << 40, 5 << 40, 7 << 40]) == INVALID


def test_binding_rejects_host_tensors():
    import torch
    x = [torch.zeros(1, 8, 8, dtype=torch.float16) for _ in range(4)]
    with pytest.raises(ValueError):
        bra.bmm_rs_a2a(x, x, None, 2, 2, 2, 4, 16, 8, 0, out=x)
    with pytest.raises(ValueError):
        bra.all_to_all_v([torch.zeros(4)] * 2, torch.zeros(2, 2, dtype=torch.int64),
                         [torch.zeros(4)] * 2, 2)
    with pytest.raises(ValueError):                  # plans check when they are made
        bra.bmm_rs_a2a_plan(x, x, None, 2, 2, 2, 4, 16, 8, 0, out=x)
    with pytest.raises(ValueError):
        bra.all_to_all_v_plan([torch.zeros(4)] * 2, torch.zeros(2, 2, dtype=torch.int64),
                              [torch.zeros(4)] * 2, 2)


def test_wait_selftest_argument_checks(lib):
    """Rejections happen on the host before any launch."""
    assert lib.bra_wait_selftest(bra.WAIT_A2AV, None, None) == NULLPTR
    assert lib.bra_wait_selftest(7, 1 << 32, None) == INVALID
    assert lib.bra_wait_selftest(-1, 1 << 32, None) == INVALID


# --------------------------------------------------------------------------
# Workspace (packed variant)
# --------------------------------------------------------------------------

def test_options_struct_layout():
    """bra_fused_options: four int32 fields (layout, variant, the two row
    pitches), the workspace pointer and its int64 size, then the per-call
    status pointer (40 bytes, 8-byte aligned)."""
    F = bra.FusedOptions
    assert ctypes.sizeof(F) == 40 and ctypes.alignment(F) == 8
    assert [getattr(F, n).offset for n in ("transpose_weight", "variant", "x_pitch", "w_pitch",
                                           "workspace", "workspace_bytes", "status")] == \
        [0, 4, 8, 12, 16, 24, 32]
    src = pathlib.Path(HEADER).read_text()
    body = src[src.index("int32_t transpose_weight;"):src.index("} bra_fused_options;")]
    decls = re.findall(r"^\s*(int32_t\*|int32_t|void\*|int64_t)\s+(\w+)", body, flags=re.M)
    assert decls == [("int32_t", "transpose_weight"), ("int32_t", "variant"),
                     ("int32_t", "x_pitch"), ("int32_t", "w_pitch"), ("void*", "workspace"),
                     ("int64_t", "workspace_bytes"), ("int32_t*", "status")]


def _ws_opts(ptr, nbytes, variant=None, transposed=False):
    o = bra._options(transposed, variant)
    o.workspace = ptr
    o.workspace_bytes = nbytes
    return o


def _ws_size(lib, f, dtype=bra.FP16, transposed=False):
    x, w, b, y = f.arrays()
    return lib.bmm_rs_a2a_workspace_size(x, w, b, *f.args, dtype, y,
                                         ctypes.byref(bra._options(transposed, None)))


def _ws_expected(f, transposed=False):
    """The documented layout restated: per rank, a copy of x when M/tp % 8 or
    its pointer is not 16-byte aligned, of the weight when its row length
    % 8 or its pointer is off; rows rounded up to 64 elements, each copy
    rounded up to 256 bytes."""
    ep, tp, E, C, M, H, t = f.args
    P, El, Kp = ep * tp, E // ep, M // tp
    if P > 1024 or any(a % 2 for a in f.x + f.w + f.y):
        return 0
    wlen = Kp if transposed else H
    px = Kp % 8 != 0 or any(a % 16 for a in f.x)
    pw = wlen % 8 != 0 or any(a % 16 for a in f.w)
    if not px and not pw:
        return 0
    r64 = lambda v: (v + 63) // 64 * 64
    r256 = lambda v: (v + 255) // 256 * 256
    xb = r256(El * ep * C * r64(Kp) * 2)
    wb = r256(El * (H if transposed else Kp) * r64(wlen) * 2)
    return P * ((xb if px else 0) + (wb if pw else 0))


@pytest.mark.parametrize("args", [(4, 2, 16, 12, 12, 4, 1), (2, 2, 4, 40, 130, 70, 0),
                                  (2, 4, 4, 260, 1028, 516, 1), (8, 2, 16, 16, 2050, 1030, 0),
                                  (2, 2, 8, 128, 128, 256, 0), (2, 2, 4, 40, 256, 70, 1),
                                  (8, 4, 64, 512, 8192, 4096, 1)])
@pytest.mark.parametrize("transposed", [False, True])
def test_workspace_size_follows_the_layout(lib, args, transposed):
    f = Fake(*args)
    assert _ws_size(lib, f, transposed=transposed) == _ws_expected(f, transposed)
    f.x[1] += 2                                   # element-aligned only: x copied
    assert _ws_size(lib, f, transposed=transposed) == _ws_expected(f, transposed)
    f.w[0] += 6
    assert _ws_size(lib, f, transposed=transposed) == _ws_expected(f, transposed) > 0
    f.y[0] += 1                                   # not element-aligned: no packed variant
    assert _ws_size(lib, f, transposed=transposed) == 0


def test_workspace_size_rejects_what_the_call_rejects(lib):
    f = Fake(2, 2, 8, 4, 8, 8, 0)
    x, w, b, y = f.arrays()
    assert lib.bmm_rs_a2a_workspace_size(x, w, b, 2, 2, 8, 4, 8, 9, 0, bra.FP16, y, None) \
        == -INVALID
    assert lib.bmm_rs_a2a_workspace_size(None, w, b, 2, 2, 8, 4, 8, 8, 0, bra.FP16, y, None) \
        == -NULLPTR
    # the workspace fields of the options are ignored by the size query
    assert lib.bmm_rs_a2a_workspace_size(x, w, b, 2, 2, 8, 4, 8, 8, 0, bra.FP16, y,
                                         ctypes.byref(_ws_opts(3, -1))) == _ws_expected(f) > 0


def test_workspace_selects_the_packed_variant(lib, monkeypatch):
    monkeypatch.delenv("BRA_FORCE_VARIANT", raising=False)
    ws = 1 << 46
    f = Fake(2, 2, 4, 40, 130, 70, 0)             # Kp = 65, H = 70: no TMA-ready rows
    need = _ws_size(lib, f)
    assert need > 0
    assert _variant(lib, f) == bra.VARIANT_TCR                              # no workspace
    assert _variant(lib, f, opts=_ws_opts(ws, need)) == bra.VARIANT_PACKED
    assert _variant(lib, f, opts=_ws_opts(ws, need - 1)) == -INVALID        # too small
    assert _variant(lib, f, opts=_ws_opts(ws + 16, need)) == -INVALID       # not 256-aligned
    assert _variant(lib, f, opts=_ws_opts(None, need)) == -INVALID          # size without memory
    assert _variant(lib, f, opts=_ws_opts(ws, -256)) == -INVALID
    assert _variant(lib, f, opts=_ws_opts(None, 0, "packed")) == -UNSUPPORTED
    assert _variant(lib, f, opts=_ws_opts(ws, need, "tcr")) == bra.VARIANT_TCR
    monkeypatch.setenv("BRA_FORCE_VARIANT", "packed")
    assert _variant(lib, f, opts=_ws_opts(ws, need)) == bra.VARIANT_PACKED
    assert _variant(lib, f) == -UNSUPPORTED
    monkeypatch.delenv("BRA_FORCE_VARIANT")
    g = Fake(8, 4, 64, 512, 8192, 4096, 1)         # TMA-ready: the workspace is not used
    assert _ws_size(lib, g) == 0
    assert _variant(lib, g, opts=_ws_opts(ws, 1 << 30)) == bra.VARIANT_TC2
    assert _variant(lib, g, opts=_ws_opts(ws, 0, "packed")) == bra.VARIANT_PACKED
    h = Fake(2, 2, 4, 40, 130, 70, 0)
    h.w[1] += 1                                   # not element-aligned: generic kernel
    assert _variant(lib, h, opts=_ws_opts(ws, 1 << 40)) == bra.VARIANT_SIMT
    assert _variant(lib, h, opts=_ws_opts(ws, 1 << 40, "packed")) == -UNSUPPORTED


def test_transposed_weight_rows_decide_tma_readiness(lib):
    """Transposed, the weight's rows are Kp long: H % 8 != 0 keeps the TMA
    kernels (ragged N reads zeros), Kp % 8 != 0 does not."""
    f = Fake(2, 2, 4, 40, 256, 70, 1)             # Kp = 128, H = 70
    assert _variant(lib, f) == bra.VARIANT_TCR
    assert _variant(lib, f, opts=bra._options(True, None)) in (bra.VARIANT_TC, bra.VARIANT_TC2)
    g = Fake(2, 2, 4, 40, 130, 64, 1)             # Kp = 65, H = 64
    assert _variant(lib, g, opts=bra._options(True, None)) == bra.VARIANT_TCR


def test_overlapping_workspace_is_rejected_before_any_launch(lib):
    f = Fake(2, 2, 4, 40, 130, 70, 0)
    need = _ws_size(lib, f)
    x, w, b, y = f.arrays()
    for base in (f.x[2] // 256 * 256, f.y[0] // 256 * 256 - 256, f.b[3] // 256 * 256):
        assert lib.bmm_rs_a2a_ex(x, w, b, *f.args, bra.FP16, y,
                                 ctypes.byref(_ws_opts(base, need)), None) == INVALID


def test_python_options_carry_the_workspace():
    """The binding passes a workspace tensor's pointer and byte size, and
    refuses one that is not a contiguous CUDA tensor."""
    import torch

    class FakeCuda:                               # stands in for a CUDA tensor on the CPU
        is_cuda = True

        def __init__(self, n, es, contiguous=True):
            self.n, self.es, self.c = n, es, contiguous

        def is_contiguous(self):
            return self.c

        def data_ptr(self):
            return 1 << 44

        def numel(self):
            return self.n

        def element_size(self):
            return self.es

    o = bra._options(True, "packed", FakeCuda(1000, 4))
    assert (o.transpose_weight, o.variant, o.workspace, o.workspace_bytes) == \
        (1, bra.VARIANT_PACKED, 1 << 44, 4000)
    assert bra._options(False, None).workspace is None
    with pytest.raises(ValueError):
        bra._options(False, None, torch.zeros(16, dtype=torch.uint8))        # a CPU tensor
    with pytest.raises(ValueError):
        bra._options(False, None, FakeCuda(16, 1, contiguous=False))


def _pitch_opts(xp=0, wp=0, variant=None, transposed=False):
    o = bra._options(transposed, variant)
    o.x_pitch, o.w_pitch = xp, wp
    return o


def test_caller_pitches_select_the_kernel_or_are_refused(lib, monkeypatch):
    """Pitched operands: a 16-byte pitch with 16-byte pointers takes the TMA
    kernels (with no workspace, H = 70 ragged); other pitches or pointers take
    the row-class kernel; what only the load-staged, generic or packed paths
    could take is BRA_ERR_UNSUPPORTED; a pitch below the row length is
    invalid."""
    monkeypatch.delenv("BRA_FORCE_VARIANT", raising=False)
    f = Fake(2, 2, 4, 40, 256, 70, 1)             # Kp = 128, H = 70: weight rows unaligned
    assert _variant(lib, f) == bra.VARIANT_TCR
    assert _variant(lib, f, opts=_pitch_opts(wp=72)) in (bra.VARIANT_TC, bra.VARIANT_TC2)
    assert _variant(lib, f, opts=_pitch_opts(xp=136, wp=80)) in (bra.VARIANT_TC, bra.VARIANT_TC2)
    assert _variant(lib, f, opts=_pitch_opts(wp=71)) == bra.VARIANT_TCR    # not a 16-byte pitch
    assert _variant(lib, f, opts=_pitch_opts(wp=69)) == -INVALID          # below the row length
    assert _variant(lib, f, opts=_pitch_opts(xp=127)) == -INVALID
    assert _variant(lib, f, opts=_pitch_opts(wp=72, variant="tcr")) == bra.VARIANT_TCR
    assert _variant(lib, f, opts=_pitch_opts(wp=72, variant="packed")) == -UNSUPPORTED
    assert _variant(lib, f, opts=_pitch_opts(wp=72, variant="tcu")) == -UNSUPPORTED
    assert _variant(lib, f, opts=_pitch_opts(wp=72, variant="simt")) == -UNSUPPORTED
    assert _variant(lib, f, opts=_pitch_opts(wp=71, variant="tc")) == -UNSUPPORTED
    assert _variant(lib, f, opts=_pitch_opts(wp=72, variant="tc")) == bra.VARIANT_TC
    assert _ws_size(lib, f) > 0
    x, w, b, y = f.arrays()
    assert lib.bmm_rs_a2a_workspace_size(x, w, b, *f.args, bra.FP16, y,
                                         ctypes.byref(_pitch_opts(wp=72))) == 0
    f.w[1] += 2                                   # element-aligned only: the row-class kernel
    assert _variant(lib, f, opts=_pitch_opts(wp=72)) == bra.VARIANT_TCR
    g = Fake(2, 16, 4, 16, 16 * 3, 5, 1)          # 8 + 8 classes x tp = 16: maps do not fit
    assert _variant(lib, g) == bra.VARIANT_TCU
    assert _variant(lib, g, opts=_pitch_opts(xp=3, wp=7)) == -UNSUPPORTED


def test_pitched_extents_enter_the_aliasing_rule(lib):
    """A pitched operand spans (rows - 1) * pitch + length elements: an
    output placed inside that span is rejected, one just past it is not."""
    f = Fake(2, 2, 4, 8, 16, 8, 0, base=1 << 41)  # x: (2, 16, 8) per rank, 32 rows of 8
    ep, tp, E, C, M, H, t = f.args
    pitch = 64
    span = ((2 * 16 - 1) * pitch + 8) * 2
    g = Fake(2, 2, 4, 8, 16, 8, 0, base=1 << 41)
    g.y[0] = g.x[0] + span - 2                    # inside the pitched span of x[0]
    assert _variant(lib, g, opts=_pitch_opts(xp=pitch)) == -INVALID
    g.y[0] = g.x[0] + ((span + 15) // 16) * 16    # 16-byte aligned, just past it
    for r in range(1, 4):                         # move the other ranks out of the way
        g.x[r] += 1 << 30
    assert _variant(lib, g, opts=_pitch_opts(xp=pitch)) > 0


def test_binding_detects_row_pitches():
    """The binding passes the shared row pitch of row-pitched x / weight
    views (0 for dense ones) and refuses other strides or mixed pitches.
    CPU tensors stand in for CUDA ones through a subclass that reports a
    CUDA device."""
    import torch

    class FakeCuda(torch.Tensor):
        @property
        def device(self):
            return torch.device("cuda", 0)

        @property
        def is_cuda(self):
            return True

    def fake(shape, pitch=None):
        d0, d1, d2 = shape
        buf = torch.zeros((d0, d1, pitch or d2), dtype=torch.float16).as_subclass(FakeCuda)
        return buf[:, :, :d2]

    shape = (2, 5, 7)
    _, p = bra._pitched_ptrs([fake(shape), fake(shape)], "x", torch.float16, shape)
    assert p == 0
    _, p = bra._pitched_ptrs([fake(shape, 9), fake(shape, 9)], "x", torch.float16, shape)
    assert p == 9
    with pytest.raises(ValueError, match="same row pitch"):
        bra._pitched_ptrs([fake(shape, 9), fake(shape, 16)], "x", torch.float16, shape)
    _, p = bra._pitched_ptrs([fake(shape), fake(shape, 7)], "x", torch.float16, shape)
    assert p == 0                                 # pitch equal to the length is dense
    odd = torch.zeros((2, 7, 5), dtype=torch.float16).as_subclass(FakeCuda).transpose(1, 2)
    with pytest.raises(ValueError, match="row-pitched"):
        bra._pitched_ptrs([odd], "x", torch.float16, shape)
    with pytest.raises(TypeError):
        bra._pitched_ptrs([fake(shape).float()], "x", torch.float16, shape)
    # d1 = 1 (ep*C = 1 rows per expert): the pitch is the step between experts.
    one = (4, 1, 6)
    _, p = bra._pitched_ptrs([fake(one, 11), fake(one, 11)], "x", torch.float16, one)
    assert p == 11
    # A pitch beyond the library's 32-bit field is refused, not wrapped.
    big = 2**31
    huge = torch.empty_strided((2, 2, 4), (2 * big, big, 1), dtype=torch.float16,
                               device="meta").as_subclass(FakeCuda)
    with pytest.raises(ValueError, match="32-bit pitch"):
        bra._pitched_ptrs([huge], "x", torch.float16, (2, 2, 4))
