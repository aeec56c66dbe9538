"""The packed variant on the GPU: operands without a 16-byte row pitch are
repacked into a caller-provided workspace (the two-phase workspace call of
the CANN guide, 调用说明), then the TMA kernel reads the copies.

* Unaligned shapes of several tiles with ragged row / column / K tails, both
  shard types, bias or not, weight stored either way: against the oracle.
* The workspace after a call holds each copied operand row for row, bit for
  bit, at the documented offsets and pitch (odd lengths padded with a zero).
* Element-aligned pointers (rows with a 16-byte pitch but starting 2..14
  bytes past a boundary) and a large shape (4100-element rows) sampled.
* A workspace filled with garbage beforehand changes nothing; a workspace
  that is too small is rejected; forcing the variant without one is refused.
"""
import numpy as np
import pytest
import torch

import bmm_reducescatter_alltoall_gb300 as bra
from oracle import fused as of
from test_fused_gpu import (TOL, UNALIGNED_CASES, _oracle, _points_check, _rel_err,
                            _sample_points, _shifted, _tile_points,
                            _to_dev)
from workloads import FUSED_CONFIGS, FusedConfig, fused_inputs_device, fused_inputs_host

pytestmark = pytest.mark.gpu


def _workspace(nbytes, fill=0xA5):
    return torch.full((max(int(nbytes), 1),), fill, dtype=torch.uint8, device="cuda")


def _call(cfg, x, w, bias, transposed, ws, variant=None):
    ys = bra.bmm_rs_a2a_infer_shape(cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H,
                                    cfg.y_shard_type)["y"]
    out = [torch.full(ys, float("nan"), dtype=x[0].dtype, device="cuda") for _ in range(cfg.P)]
    bra.bmm_rs_a2a(x, w, bias, cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, cfg.y_shard_type,
                   out=out, transpose_weight=transposed, variant=variant, workspace=ws)
    torch.cuda.synchronize()
    assert bra.fault_status() == 0
    return out


def _need(cfg, x, w, bias, transposed):
    ys = bra.bmm_rs_a2a_infer_shape(cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H,
                                    cfg.y_shard_type)["y"]
    probe = [torch.empty(ys, dtype=x[0].dtype, device="cuda") for _ in range(cfg.P)]
    return bra.bmm_rs_a2a_workspace_size(x, w, bias, cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M,
                                         cfg.H, cfg.y_shard_type, probe,
                                         transpose_weight=transposed), probe


@pytest.mark.parametrize("transposed", [False, True])
@pytest.mark.parametrize("case", UNALIGNED_CASES)
@pytest.mark.parametrize("bias", [True, False])
def test_packed_unaligned_shapes(case, bias, transposed):
    ep, tp, E, C, M, H, t, dt = case
    cfg = FusedConfig("pk", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=sum(case[:6]) + 23, has_bias=bias)
    inp = fused_inputs_host(cfg)
    ref = _oracle(cfg, inp)
    d = _to_dev(inp)
    w = [u.transpose(1, 2).contiguous() for u in d["w"]] if transposed else d["w"]
    need, probe = _need(cfg, d["x"], w, d["bias"], transposed)
    assert need > 0
    ws = _workspace(need)
    assert bra.bmm_rs_a2a_variant(d["x"], w, d["bias"], ep, tp, E, C, M, H, t, probe,
                                  transpose_weight=transposed, workspace=ws) == \
        bra.VARIANT_PACKED
    out = _call(cfg, d["x"], w, d["bias"], transposed, ws)
    err = _rel_err(out, ref)
    assert err <= TOL[dt], f"{case} bias={bias} transposed={transposed}: rel err {err:.3e}"


def _r64(v):
    return (v + 63) // 64 * 64


def _r256(v):
    return (v + 255) // 256 * 256


@pytest.mark.parametrize("transposed", [False, True])
@pytest.mark.parametrize("case", [(2, 2, 4, 40, 130, 70, 0, "fp16"),
                                  (4, 4, 8, 33 * 4, 36, 4, 1, "bf16"),
                                  (2, 4, 4, 260, 1028, 516, 1, "fp16")])
def test_workspace_holds_the_repacked_rows(case, transposed):
    """x copies of every rank first, then weight copies; rows `pitch`
    elements apart; each copy 256-byte aligned; bit-exact."""
    ep, tp, E, C, M, H, t, dt = case
    cfg = FusedConfig("pkw", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=sum(case[:6]))
    d = _to_dev(fused_inputs_host(cfg))
    w = [u.transpose(1, 2).contiguous() for u in d["w"]] if transposed else d["w"]
    need, _ = _need(cfg, d["x"], w, d["bias"], transposed)
    ws = _workspace(need)
    _call(cfg, d["x"], w, d["bias"], transposed, ws)
    P, El, Kp = cfg.P, E // ep, M // tp
    wlen = Kp if transposed else H
    wrows = El * (H if transposed else Kp)
    xrows = El * ep * C
    xb, wb = _r256(xrows * _r64(Kp) * 2), _r256(wrows * _r64(wlen) * 2)
    px, pw = Kp % 8 != 0, wlen % 8 != 0
    assert need == P * ((xb if px else 0) + (wb if pw else 0))
    raw = ws.cpu()
    off = 0
    for copied, srcs, nb, rows, length in ((px, d["x"], xb, xrows, Kp), (pw, w, wb, wrows, wlen)):
        if not copied:
            continue
        for r in range(P):
            blk = raw[off:off + rows * _r64(length) * 2].view(torch.int16).view(rows, _r64(length))
            want = srcs[r].reshape(rows, length).view(torch.int16).cpu()
            assert torch.equal(blk[:, :length], want), f"rank {r}"
            if length % 2:
                assert (blk[:, length] == 0).all()
            off += nb


@pytest.mark.parametrize("transposed", [False, True])
def test_packed_element_aligned_pointers(transposed):
    """Rows with a 16-byte pitch whose tensors start 1..7 elements past a
    boundary: only the misplaced operands are copied."""
    M, H = 272, 264
    cfg = FusedConfig("pkp", ep=4, tp=2, E=8, C=96, M=M, H=H, y_shard_type=1, dtype="bf16",
                      seed=M + H + 1)
    inp = fused_inputs_host(cfg)
    ref = _oracle(cfg, inp)
    d = _to_dev(inp)
    xs = [_shifted(x, 1 + r % 7) for r, x in enumerate(d["x"])]
    w0 = [u.transpose(1, 2).contiguous() for u in d["w"]] if transposed else d["w"]
    need_w_only, _ = _need(cfg, d["x"], [_shifted(u, 3) for u in w0], d["bias"], transposed)
    need, _ = _need(cfg, xs, w0, d["bias"], transposed)
    assert 0 < need and 0 < need_w_only
    out = _call(cfg, xs, w0, d["bias"], transposed, _workspace(need))
    err = _rel_err(out, ref)
    assert err <= TOL["bf16"], f"transposed={transposed}: rel err {err:.3e}"


@pytest.mark.parametrize("transposed", [False, True])
def test_packed_large_every_tile(transposed):
    """4100-element token and weight rows (8200-byte pitch), 16 ranks, both
    operands copied; a point in every output tile against the oracle."""
    cfg = FUSED_CONFIGS["ep8tp2_E64_C256_M4096_H4096_t0_bf16"].replace(E=16, M=4100, H=4100)
    dinp = fused_inputs_device(cfg)
    w = [u.transpose(1, 2).contiguous() for u in dinp["w"]] if transposed else dinp["w"]
    need, _ = _need(cfg, dinp["x"], w, dinp["bias"], transposed)
    out = _call(cfg, dinp["x"], w, dinp["bias"], transposed, _workspace(need))
    for y in out:
        assert not torch.isnan(y).any().item()
    rng = np.random.default_rng(13)
    err = _points_check(cfg, dinp, out, _tile_points(cfg, rng) + _sample_points(cfg, rng, 4))
    assert err <= TOL["bf16"], f"rel err {err:.3e}"


def test_workspace_contents_do_not_matter_and_calls_repeat_bit_identically():
    cfg = FusedConfig("pkr", ep=4, tp=2, E=8, C=160, M=1026, H=518, y_shard_type=0,
                      dtype="bf16", seed=5)
    d = _to_dev(fused_inputs_host(cfg))
    need, _ = _need(cfg, d["x"], d["w"], d["bias"], False)
    outs = [_call(cfg, d["x"], d["w"], d["bias"], False, _workspace(need, fill))
            for fill in (0, 0xFF, 0x7C)]
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_small_workspace_and_forced_variant_are_refused(monkeypatch):
    monkeypatch.delenv("BRA_FORCE_VARIANT", raising=False)
    cfg = FusedConfig("pks", ep=2, tp=2, E=4, C=40, M=130, H=70, y_shard_type=0, dtype="fp16",
                      seed=3)
    d = _to_dev(fused_inputs_host(cfg))
    need, probe = _need(cfg, d["x"], d["w"], d["bias"], False)
    with pytest.raises(bra.BraError) as e:
        _call(cfg, d["x"], d["w"], d["bias"], False, _workspace(need - 256))
    assert e.value.args[0].endswith(f"({bra.ERR_INVALID})")
    with pytest.raises(bra.BraError) as e:
        _call(cfg, d["x"], d["w"], d["bias"], False, None, variant="packed")
    assert e.value.args[0].endswith(f"({bra.ERR_UNSUPPORTED})")
    # an aligned shape ignores the workspace; forced, the packed variant
    # copies nothing and runs the TMA kernel on the caller's tensors
    cfg2 = cfg.replace(M=256, H=512)
    inp2 = fused_inputs_host(cfg2)
    d2 = _to_dev(inp2)
    assert _need(cfg2, d2["x"], d2["w"], d2["bias"], False)[0] == 0
    out = _call(cfg2, d2["x"], d2["w"], d2["bias"], False, None, variant="packed")
    assert _rel_err(out, _oracle(cfg2, inp2)) <= TOL["fp16"]


@pytest.mark.parametrize("case", [
    (32, 32, 32, 2, 32 * 6, 32 * 5, 0, "fp16"),   # P = 1024: 2048 copies, eight repack launches
    (2, 1, 2, 2, 16, 65535, 0, "bf16"),           # weight rows of 65535 elements (pitch 65536)
    (2, 1, 2, 2, 65535, 16, 1, "fp16"),           # x rows of 65535 elements, 1024 K blocks
])
def test_packed_at_the_limits(case):
    ep, tp, E, C, M, H, t, dt = case
    cfg = FusedConfig("pkl", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=ep + tp + E + C + 1)
    inp = fused_inputs_host(cfg)
    ref = _oracle(cfg, inp)
    d = _to_dev(inp)
    need, probe = _need(cfg, d["x"], d["w"], d["bias"], False)
    ws = _workspace(need)
    assert bra.bmm_rs_a2a_variant(d["x"], d["w"], d["bias"], ep, tp, E, C, M, H, t, probe,
                                  workspace=ws) == bra.VARIANT_PACKED
    out = _call(cfg, d["x"], d["w"], d["bias"], False, ws)
    err = _rel_err(out, ref)
    assert err <= TOL[dt], f"{case}: rel err {err:.3e}"


def test_auto_workspace():
    """workspace="auto": the binding takes the size the library asks for from
    torch's allocator (none for TMA-ready operands) and the packed variant runs."""
    cfg = FusedConfig("pka", ep=2, tp=2, E=4, C=40, M=130, H=70, y_shard_type=0, dtype="fp16",
                      seed=9)
    inp = fused_inputs_host(cfg)
    d = _to_dev(inp)
    plan = bra.bmm_rs_a2a_plan(d["x"], d["w"], d["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M,
                               cfg.H, cfg.y_shard_type, workspace="auto")
    ws = plan._keep[-1]
    need, _ = _need(cfg, d["x"], d["w"], d["bias"], False)
    assert ws is not None and ws.numel() == need
    out = plan.run()
    torch.cuda.synchronize()
    assert bra.fault_status() == 0
    assert _rel_err(out, _oracle(cfg, inp)) <= TOL["fp16"]
    cfg2 = cfg.replace(M=256, H=512)
    d2 = _to_dev(fused_inputs_host(cfg2))
    plan2 = bra.bmm_rs_a2a_plan(d2["x"], d2["w"], d2["bias"], cfg2.ep, cfg2.tp, cfg2.E, cfg2.C,
                                cfg2.M, cfg2.H, cfg2.y_shard_type, workspace="auto")
    assert plan2._keep[-1] is None
    with pytest.raises(ValueError):
        bra.bmm_rs_a2a(d2["x"], d2["w"], d2["bias"], cfg2.ep, cfg2.tp, cfg2.E, cfg2.C, cfg2.M,
                       cfg2.H, cfg2.y_shard_type, workspace="big")


def _padded_view(t, pitch, offset=0):
    """A (d0, d1, pitch) buffer whose padding holds NaN, viewed as t's shape
    and holding t's values: a row-pitched operand.  With an offset the view
    starts that many elements into its buffer (a base address without
    16-byte alignment)."""
    d0, d1, d2 = t.shape
    buf = torch.full((offset + d0 * d1 * pitch,), float("nan"), dtype=t.dtype, device=t.device)
    v = buf.as_strided((d0, d1, d2), (d1 * pitch, pitch, 1), offset)
    v.copy_(t)
    return v


@pytest.mark.parametrize("case,xpitch,wpitch,transposed", [
    ((2, 2, 4, 40, 256, 70, 1, "fp16"), 0, 72, False),     # H = 70: only the weight pitched
    ((2, 2, 4, 40, 130, 70, 0, "bf16"), 72, 80, False),    # Kp = 65 and H = 70 both pitched
    ((4, 2, 8, 96, 200, 300, 1, "fp16"), 104, 0, True),    # transposed weight, rows of Kp = 100
    ((2, 2, 4, 40, 130, 70, 0, "bf16"), 67, 73, False),    # odd pitches: the row-class kernel
    ((2, 2, 4, 6, 12, 4, 1, "fp16"), 7, 5, False),         # rows of 6 and 4 elements, pitches 7, 5
    ((4, 2, 8, 96, 200, 300, 1, "bf16"), 103, 0, True),    # transposed, odd pitch
])
def test_caller_pitched_operands(case, xpitch, wpitch, transposed):
    _pitched_case(case, xpitch, wpitch, transposed, 0, 0)


@pytest.mark.parametrize("case,xpitch,wpitch,xoff,woff", [
    ((2, 2, 4, 6, 12, 4, 1, "fp16"), 7, 5, 1, 3),          # rows of 6 and 4, odd pitches
    ((2, 2, 4, 6, 12, 4, 0, "bf16"), 7, 5, 5, 7),
    ((2, 2, 4, 40, 130, 70, 0, "bf16"), 67, 73, 2, 6),     # Kp = 65 and H = 70
    ((2, 2, 4, 40, 256, 70, 1, "fp16"), 0, 71, 0, 1),      # only the weight pitched
])
def test_caller_pitched_operands_unaligned_base(case, xpitch, wpitch, xoff, woff):
    """Row-pitched views that start 1..7 elements into their buffers: base
    addresses without 16-byte alignment reach the row-class kernel (short
    rows included) and match the oracle; the padding is never read."""
    _pitched_case(case, xpitch, wpitch, False, xoff, woff)


def _pitched_case(case, xpitch, wpitch, transposed, xoff, woff):
    """Operands kept in padded buffers run with no copy and no workspace:
    16-byte pitches on the TMA kernels, other pitches on the row-class
    kernel; the padding (NaN) is never read."""
    ep, tp, E, C, M, H, t, dt = case
    cfg = FusedConfig("pit", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=sum(case[:6]) + 31)
    inp = fused_inputs_host(cfg)
    ref = _oracle(cfg, inp)
    d = _to_dev(inp)
    w0 = [u.transpose(1, 2).contiguous() for u in d["w"]] if transposed else d["w"]
    if transposed:
        xs = [_padded_view(x, xpitch) for x in d["x"]]
        ws = [_padded_view(u, xpitch) for u in w0]          # transposed rows are Kp long too
    else:
        xs = [_padded_view(x, xpitch, xoff) for x in d["x"]] if xpitch else d["x"]
        ws = [_padded_view(u, wpitch, woff) for u in w0] if wpitch else w0
    ys = bra.bmm_rs_a2a_infer_shape(ep, tp, E, C, M, H, t)["y"]
    probe = [torch.empty(ys, dtype=xs[0].dtype, device="cuda") for _ in range(cfg.P)]
    pitches = [p for p in (xpitch, wpitch) if p]
    aligned = all(p % 8 == 0 for p in pitches) and xoff % 8 == 0 and woff % 8 == 0
    want = (bra.VARIANT_TC, bra.VARIANT_TC2) if aligned else (bra.VARIANT_TCR,)
    assert bra.bmm_rs_a2a_variant(xs, ws, d["bias"], ep, tp, E, C, M, H, t, probe,
                                  transpose_weight=transposed) in want
    assert bra.bmm_rs_a2a_workspace_size(xs, ws, d["bias"], ep, tp, E, C, M, H, t, probe,
                                         transpose_weight=transposed) == 0
    out = _call(cfg, xs, ws, d["bias"], transposed, None)
    err = _rel_err(out, ref)
    assert err <= TOL[dt], f"{case}: rel err {err:.3e}"
