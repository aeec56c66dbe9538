"""Fused BMM -> ReduceScatter -> Add -> AllToAll on the GPU against the oracle.

Tolerance: max|gpu - oracle| / max|oracle| <= 2e-3 for fp16 and 1e-2 for
bf16, over every output element (small shapes); at the full-size workloads
over every output element of six whole sender groups (s, e), and over a
point in every 128 x 256 output tile of every group, computed one by one by
the oracle.  Every case is
also run without bias, so the bias (N(0,1), the largest term at the full
sizes) cannot hide an error in the contraction.
"""
import numpy as np
import pytest
import torch

import bmm_reducescatter_alltoall_gb300 as bra
from oracle import fused as of
from workloads import FUSED_CONFIGS, FusedConfig, fused_inputs_device, fused_inputs_host

pytestmark = pytest.mark.gpu

TOL = {"fp16": 2e-3, "bf16": 1e-2}


def _to_dev(inp):
    return {k: (None if v is None else [t.cuda() for t in v]) for k, v in inp.items()}


def _run(cfg, dinp, variant=None, monkeypatch=None, prefill_nan=True):
    dt = torch.float16 if cfg.dtype == "fp16" else torch.bfloat16
    ys = bra.bmm_rs_a2a_infer_shape(cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H,
                                    cfg.y_shard_type)["y"]
    out = [torch.full(ys, float("nan") if prefill_nan else 0.0, dtype=dt, device="cuda")
           for _ in range(cfg.P)]
    if monkeypatch is not None:
        if variant:
            monkeypatch.setenv("BRA_FORCE_VARIANT", variant)
        else:
            monkeypatch.delenv("BRA_FORCE_VARIANT", raising=False)
    bra.bmm_rs_a2a(dinp["x"], dinp["w"], dinp["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M,
                   cfg.H, cfg.y_shard_type, out=out)
    torch.cuda.synchronize()
    assert bra.fault_status() == 0
    return out


def _rel_err(gpu, ref):
    g = np.concatenate([a.float().cpu().numpy().astype(np.float64).ravel() for a in gpu])
    r = np.concatenate([a.ravel() for a in ref])
    assert np.isfinite(g).all(), "an output element was not written"
    return float(np.max(np.abs(g - r)) / max(np.max(np.abs(r)), 1e-30))


def _oracle(cfg, inp):
    return of.bmm_rs_a2a(inp["x"], inp["w"], inp["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M,
                         cfg.H, cfg.y_shard_type, cfg.dtype)


def _check_small(cfg, monkeypatch, variant=None, bias_ndim=3):
    inp = fused_inputs_host(cfg, bias_ndim=bias_ndim)
    ref = _oracle(cfg, inp)
    out = _run(cfg, _to_dev(inp), variant, monkeypatch)
    err = _rel_err(out, ref)
    assert err <= TOL[cfg.dtype], f"{cfg} variant={variant}: rel err {err:.3e}"
    return out, ref


def test_eight_rank_example(monkeypatch):
    cfg = FUSED_CONFIGS["ep4tp2_E16_C12_M12_H4_t1_fp16"]
    _check_small(cfg, monkeypatch)
    _check_small(cfg.replace(has_bias=False), monkeypatch)
    _check_small(cfg, monkeypatch, bias_ndim=2)
    # the same example with the H-sharded layout
    _check_small(cfg.replace(y_shard_type=0), monkeypatch)


# Shapes the tensor-core kernel takes, with ragged row / column / K tails.
TC_CASES = [
    # ep, tp, E, C, M, H, type, dtype
    (2, 2, 4, 96, 256, 512, 0, "fp16"),
    (4, 2, 8, 40, 208, 328, 1, "bf16"),
    (1, 1, 2, 130, 72, 264, 0, "fp16"),
    (2, 1, 4, 64, 64, 256, 1, "bf16"),
    (8, 4, 16, 64, 256, 256, 1, "fp16"),
    (4, 4, 8, 128, 512, 512, 0, "bf16"),
    (8, 8, 8, 16, 128, 128, 0, "fp16"),       # P = 64
    (16, 8, 16, 8, 64, 128, 0, "bf16"),       # P = 128: two launches
    (2, 4, 4, 200, 96, 40, 1, "fp16"),        # H = 40 < one column tile
    (2, 2, 2, 1, 16, 16, 0, "fp16"),          # one token
    (2, 2, 4, 64, 128, 2056, 1, "bf16"),
    (2, 2, 4, 64, 6144, 2056, 1, "bf16"),     # 512-wide pair tiles (long K), ragged last tile
    (2, 4, 4, 32, 8192, 512, 0, "fp16"),      # 512-wide pair tiles, tp = 4
]


_WANT = {"tc": bra.VARIANT_TC, "tc2": bra.VARIANT_TC2, "tcu": bra.VARIANT_TCU,
         "tcr": bra.VARIANT_TCR, "simt": bra.VARIANT_SIMT}


@pytest.mark.parametrize("variant", ["tc", "tc2", "tcr", "tcu"])
@pytest.mark.parametrize("case", TC_CASES)
@pytest.mark.parametrize("bias", [True, False])
def test_tensor_core_kernels(case, bias, variant, monkeypatch):
    ep, tp, E, C, M, H, t, dt = case
    cfg = FusedConfig("tc", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=sum(case[:6]), has_bias=bias)
    inp = fused_inputs_host(cfg)
    dinp = _to_dev(inp)
    ys = bra.bmm_rs_a2a_infer_shape(ep, tp, E, C, M, H, t)["y"]
    probe = [torch.empty(ys, dtype=dinp["x"][0].dtype, device="cuda") for _ in range(cfg.P)]
    monkeypatch.setenv("BRA_FORCE_VARIANT", variant)
    want = _WANT[variant]
    assert bra.bmm_rs_a2a_variant(dinp["x"], dinp["w"], dinp["bias"], ep, tp, E, C, M, H, t,
                                  probe) == want
    ref = _oracle(cfg, inp)
    out = _run(cfg, dinp, variant, monkeypatch)
    err = _rel_err(out, ref)
    assert err <= TOL[dt], f"{case} bias={bias} {variant}: rel err {err:.3e}"


@pytest.mark.parametrize("case", TC_CASES)
@pytest.mark.parametrize("bias", [True, False])
def test_pair_kernel_wide_tiles(case, bias, monkeypatch, capfd):
    """The CTA-pair kernel with 256 x 512 tiles forced (eight epilogue warps,
    one accumulator per CTA) on every shape of the table, against the oracle."""
    ep, tp, E, C, M, H, t, dt = case
    cfg = FusedConfig("tcw", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=sum(case[:6]) + 41, has_bias=bias)
    inp = fused_inputs_host(cfg)
    ref = _oracle(cfg, inp)
    monkeypatch.setenv("BRA_TC2_WIDE", "1")
    monkeypatch.setenv("BRA_LOG", "1")
    capfd.readouterr()
    out = _run(cfg, _to_dev(inp), "tc2", monkeypatch)
    assert "-> tc2 (256x512 tiles)" in capfd.readouterr().err
    err = _rel_err(out, ref)
    assert err <= TOL[dt], f"{case} bias={bias}: rel err {err:.3e}"


@pytest.mark.parametrize("wide", ["0", "1"])
@pytest.mark.parametrize("case", TC_CASES + [(4, 4, 8, 264, 8192, 1104, 0, "bf16"),
                                             (2, 2, 4, 300, 512, 1024, 1, "fp16")])
def test_pair_kernel_shared_weight_boxes(case, wide, monkeypatch, capfd):
    """Two CTA pairs per cluster computing m tiles 2i and 2i+1 of one n tile,
    each weight box loaded once and multicast to both pairs (odd m-tile counts
    leave the second pair a tile past the rows), both tile widths, against the
    oracle."""
    ep, tp, E, C, M, H, t, dt = case
    cfg = FusedConfig("tcs", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=sum(case[:6]) + 47)
    inp = fused_inputs_host(cfg)
    ref = _oracle(cfg, inp)
    monkeypatch.setenv("BRA_TC2_SHARE", "1")
    monkeypatch.setenv("BRA_TC2_WIDE", wide)
    monkeypatch.setenv("BRA_LOG", "1")
    capfd.readouterr()
    out = _run(cfg, _to_dev(inp), "tc2", monkeypatch)
    assert "weight boxes shared)" in capfd.readouterr().err
    err = _rel_err(out, ref)
    assert err <= TOL[dt], f"{case} wide={wide}: rel err {err:.3e}"


@pytest.mark.parametrize("case,wide", [
    ((4, 4, 8, 256, 8192, 1024, 1, "fp16"), True),    # K = 8192, H = 1024: 64 wide tiles
    ((4, 4, 8, 264, 8192, 1104, 0, "bf16"), True),    # ragged m and n tiles, H/tp = 276
    ((4, 2, 8, 256, 4096, 1024, 0, "bf16"), False),   # K = 4096: 256-wide
    ((4, 4, 8, 256, 8192, 512, 1, "fp16"), False),    # H < 1024: 256-wide
])
def test_pair_kernel_tile_width_choice(case, wide, monkeypatch, capfd):
    """The automatic choice of the pair tile's width follows the K loop's
    length, H and the tile count, and both widths match the oracle."""
    ep, tp, E, C, M, H, t, dt = case
    cfg = FusedConfig("tcx", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=sum(case[:6]) + 43)
    inp = fused_inputs_host(cfg)
    ref = _oracle(cfg, inp)
    monkeypatch.delenv("BRA_TC2_WIDE", raising=False)
    monkeypatch.setenv("BRA_LOG", "1")
    capfd.readouterr()
    out = _run(cfg, _to_dev(inp), None, monkeypatch)
    log = capfd.readouterr().err
    assert ("-> tc2 (256x512 tiles)" if wide else "-> tc2 (256x256 tiles)") in log, log
    err = _rel_err(out, ref)
    assert err <= TOL[dt], f"{case}: rel err {err:.3e}"


@pytest.mark.parametrize("case", TC_CASES[:5])
def test_generic_kernel_on_the_same_shapes(case, monkeypatch):
    ep, tp, E, C, M, H, t, dt = case
    cfg = FusedConfig("simt", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=sum(case[:6]) + 1)
    _check_small(cfg, monkeypatch, variant="simt")


@pytest.mark.parametrize("case", [
    (2, 2, 4, 6, 12, 10, 0, "fp16"),      # H/tp = 5: unaligned rows
    (4, 2, 8, 12, 14, 4, 1, "bf16"),      # M/tp = 7
    (2, 1, 2, 3, 5, 7, 1, "fp16"),
    (4, 4, 8, 8, 20, 36, 0, "bf16"),
])
@pytest.mark.parametrize("variant", [None, "tcu", "simt"])
def test_unaligned_shapes_small(case, variant, monkeypatch):
    """Rows without a 16-byte pitch: the row-class TMA kernel (the automatic
    choice), the load-staged tensor-core kernel and the generic kernel."""
    ep, tp, E, C, M, H, t, dt = case
    cfg = FusedConfig("u", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=sum(case[:6]) + 2)
    _check_small(cfg, monkeypatch, variant=variant)
    _check_small(cfg.replace(has_bias=False), monkeypatch, variant=variant)


# Unaligned shapes over several tiles, with ragged row / column / K tails:
# K per shard, H or H/tp not a multiple of 8 elements.
UNALIGNED_CASES = [
    # ep, tp, E, C, M, H, type, dtype
    (2, 2, 4, 40, 130, 70, 0, "fp16"),        # Kp = 65, H/tp = 35
    (2, 2, 4, 40, 130, 70, 1, "bf16"),
    (4, 2, 8, 96, 200, 300, 0, "bf16"),       # Kp = 100 (200-byte rows), 3 m-tiles, 2 n-tiles
    (2, 4, 4, 260, 1028, 516, 1, "fp16"),     # Kp = 257, ragged 5 m-tiles x 3 n-tiles
    (4, 4, 8, 33 * 4, 36, 4, 1, "fp16"),      # Kp = 9, H = 4: K and N far below one block
    (8, 2, 16, 16, 2050, 1030, 0, "bf16"),    # P = 16, Kp = 1025, H/tp = 515
]


@pytest.mark.parametrize("variant", [None, "tcu"])
@pytest.mark.parametrize("case", UNALIGNED_CASES)
@pytest.mark.parametrize("bias", [True, False])
def test_unaligned_shapes_tensor_core(case, bias, variant, monkeypatch):
    ep, tp, E, C, M, H, t, dt = case
    cfg = FusedConfig("ut", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=sum(case[:6]) + 11, has_bias=bias)
    inp = fused_inputs_host(cfg)
    dinp = _to_dev(inp)
    ys = bra.bmm_rs_a2a_infer_shape(ep, tp, E, C, M, H, t)["y"]
    probe = [torch.empty(ys, dtype=dinp["x"][0].dtype, device="cuda") for _ in range(cfg.P)]
    monkeypatch.delenv("BRA_FORCE_VARIANT", raising=False)
    assert bra.bmm_rs_a2a_variant(dinp["x"], dinp["w"], dinp["bias"], ep, tp, E, C, M, H, t,
                                  probe) == bra.VARIANT_TCR
    ref = _oracle(cfg, inp)
    out = _run(cfg, dinp, variant, monkeypatch)
    err = _rel_err(out, ref)
    assert err <= TOL[dt], f"{case} bias={bias} {variant}: rel err {err:.3e}"


def test_unaligned_2d_bias_and_generic_agree(monkeypatch):
    cfg = FusedConfig("u2", ep=4, tp=2, E=8, C=96, M=200, H=300, y_shard_type=1, dtype="fp16",
                      seed=21)
    _check_small(cfg, monkeypatch, bias_ndim=2)
    dinp = _to_dev(fused_inputs_host(cfg))
    b = _run(cfg, dinp, "simt", monkeypatch)
    ref = [u.float().cpu().numpy().astype(np.float64) for u in b]
    for v in ("tcr", "tcu"):
        a = _run(cfg, dinp, v, monkeypatch)
        assert _rel_err(a, ref) <= TOL["fp16"], v


@pytest.mark.parametrize("variant", ["tc", "tc2", "tcr", "tcu"])
def test_tc_and_generic_agree(variant, monkeypatch):
    cfg = FusedConfig("x", ep=4, tp=2, E=8, C=128, M=256, H=512, y_shard_type=1,
                      dtype="bf16", seed=3)
    dinp = _to_dev(fused_inputs_host(cfg))
    a = _run(cfg, dinp, variant, monkeypatch)
    b = _run(cfg, dinp, "simt", monkeypatch)
    ref = [t.float().cpu().numpy().astype(np.float64) for t in b]
    assert _rel_err(a, ref) <= TOL["bf16"]


# --------------------------------------------------------------------------
# Full-size workloads: whole expert blocks, and a point in every tile
# --------------------------------------------------------------------------

def _sample_points(cfg, rng, per_rank=24):
    ys = of.infer_shapes(cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, cfg.y_shard_type)["y"]
    pts = []
    for d in range(cfg.P):
        edge = [(0, 0, 0), (ys[0] - 1, ys[1] - 1, ys[2] - 1),
                (int(rng.integers(ys[0])), min(127, ys[1] - 1), min(255, ys[2] - 1)),
                (int(rng.integers(ys[0])), min(128, ys[1] - 1), min(256, ys[2] - 1))]
        pts += [(d,) + p for p in edge]
        for _ in range(per_rank - len(edge)):
            pts.append((d, int(rng.integers(ys[0])), int(rng.integers(ys[1])),
                        int(rng.integers(ys[2]))))
    return pts


def _tile_points(cfg, rng, tile_m=128, tile_n=256):
    """One random point inside every tile_m x tile_n tile of every sender
    group's tp-summed product Z_{s,e} (ep*C x H), as output coordinates
    (d, i, c, h).  128 x 256 tiles refine both kernels' tilings (128 x 256
    one-CTA tiles, 256 x 256 pair tiles), so a tile computed from the wrong
    group, band or shard, or stored to the wrong place, shows at a point."""
    El, rows = cfg.E // cfg.ep, cfg.ep * cfg.C
    mts, nts = -(-rows // tile_m), -(-cfg.H // tile_n)
    g, mt, nt = np.meshgrid(np.arange(cfg.ep * El), np.arange(mts), np.arange(nts),
                            indexing="ij")
    g, mt, nt = g.ravel(), mt.ravel(), nt.ravel()
    zrow = mt * tile_m + rng.integers(0, np.minimum(tile_m, rows - mt * tile_m))
    zcol = nt * tile_n + rng.integers(0, np.minimum(tile_n, cfg.H - nt * tile_n))
    s, e = g // El, g % El
    j = zrow // cfg.C
    if cfg.y_shard_type == 0:
        Hp = cfg.H // cfg.tp
        t, c, h = zcol // Hp, zrow % cfg.C, zcol % Hp
    else:
        Cp = cfg.C // cfg.tp
        t, c, h = (zrow % cfg.C) // Cp, (zrow % cfg.C) % Cp, zcol
    return list(zip((j * cfg.tp + t).tolist(), (s * El + e).tolist(), c.tolist(), h.tolist(),
                    zrow.tolist(), zcol.tolist()))


def _points_check(cfg, dinp, out, pts, w_transposed=False):
    """max|gpu - oracle| / max|oracle| over output points (d, i, c, h, ...),
    each evaluated by the oracle's receiver view: its source found by
    y_source, then the tp dot products of one x row and one weight column
    plus the sender's bias, rounded once."""
    El = cfg.E // cfg.ep
    src = [of.y_source(cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.H, cfg.y_shard_type, *p[:4])
           for p in pts]
    for p, q in zip(pts, src):                 # the points were aimed at these Z entries
        if len(p) > 4:
            assert (q["zrow"], q["zcol"]) == (p[4], p[5]), (p, q)
    dev = dinp["x"][0].device
    got = np.empty(len(pts))
    want = np.empty(len(pts))
    by_d, by_s = {}, {}
    for k, (p, q) in enumerate(zip(pts, src)):
        by_d.setdefault(p[0], []).append(k)
        by_s.setdefault(q["s"], []).append(k)
    for d, ks in by_d.items():
        idx = [torch.tensor([pts[k][a] for k in ks], device=dev) for a in (1, 2, 3)]
        got[ks] = out[d][idx[0], idx[1], idx[2]].double().cpu().numpy()
    for s, ks in by_s.items():
        e = torch.tensor([src[k]["e"] for k in ks], device=dev)
        zr = torch.tensor([src[k]["zrow"] for k in ks], device=dev)
        zc = torch.tensor([src[k]["zcol"] for k in ks], device=dev)
        ranks = [s * cfg.tp + u for u in range(cfg.tp)]
        rows = torch.stack([dinp["x"][r][e, zr, :] for r in ranks], 1).double().cpu().numpy()
        cols = torch.stack([(dinp["w"][r][e, zc, :] if w_transposed else dinp["w"][r][e, :, zc])
                            for r in ranks], 1).double().cpu().numpy()
        for n, k in enumerate(ks):
            b = None
            if dinp["bias"] is not None:
                q = src[k]
                b = float(dinp["bias"][q["bias_rank"]].reshape(El, -1)[q["e"], q["bias_col"]])
            want[k] = of.bmm_rs_a2a_point(rows[n], cols[n], b, cfg.dtype)
    assert np.isfinite(got).all(), "an output element was not written"
    return float(np.max(np.abs(got - want)) / np.max(np.abs(want)))


FULL_SIZE = ["ep8tp2_E64_C256_M4096_H4096_t0_bf16", "ep8tp4_E64_C512_M8192_H4096_t1_fp16"]


@pytest.mark.parametrize("variant", [None, "tc", "tc2"])
@pytest.mark.parametrize("name", FULL_SIZE)
def test_full_size_workloads_every_tile(name, variant, monkeypatch):
    """A point in every 128 x 256 output tile of every (rank, expert) group,
    plus the tile-seam points of every receiver, against the oracle."""
    cfg = FUSED_CONFIGS[name]
    rng = np.random.default_rng(99)
    for bias in (True, False):
        c = cfg.replace(has_bias=bias)
        dinp = fused_inputs_device(c)
        out = _run(c, dinp, variant, monkeypatch)
        for y in out:                                  # every element written
            assert not torch.isnan(y).any().item()
        pts = _tile_points(c, rng) + _sample_points(c, rng, per_rank=4)
        err = _points_check(c, dinp, out, pts)
        assert err <= TOL[cfg.dtype], f"{name} bias={bias}: rel err {err:.3e} at {len(pts)} points"
        del dinp, out
        torch.cuda.empty_cache()


# Sender groups (s, e) compared whole: the first and the last group of the
# launch (the last one ends in a partial wave of CTA pairs), and groups whose
# tiles start at different offsets into a wave.
WHOLE_GROUPS = [(0, 0), (1, 3), (3, 7), (5, 1), (6, 6), (7, 7)]


@pytest.mark.parametrize("name", FULL_SIZE)
def test_full_size_whole_expert_blocks(name, monkeypatch):
    """Every output element that six whole sender groups (s, e) produce --
    their blocks at all ep*tp receivers -- against the oracle's evaluation of
    those groups, with and without bias, on the kernel the bench times."""
    cfg = FUSED_CONFIGS[name]
    El, tp = cfg.E // cfg.ep, cfg.tp
    for bias in (True, False):
        c = cfg.replace(has_bias=bias)
        dinp = fused_inputs_device(c)
        out = _run(c, dinp, None, monkeypatch)
        num = den = 0.0
        n = 0
        for s, e in WHOLE_GROUPS:
            ranks = [s * tp + u for u in range(tp)]
            bg = None if not bias else [dinp["bias"][r].reshape(El, -1)[e].cpu() for r in ranks]
            blocks = of.group_outputs([dinp["x"][r][e].cpu() for r in ranks],
                                      [dinp["w"][r][e].cpu() for r in ranks], bg,
                                      c.ep, tp, c.C, c.H, c.y_shard_type, c.dtype)
            for (j, u), ref in blocks.items():
                got = out[j * tp + u][s * El + e].double().cpu().numpy()
                assert np.isfinite(got).all(), "an output element was not written"
                num = max(num, float(np.max(np.abs(got - ref))))
                den = max(den, float(np.max(np.abs(ref))))
                n += ref.size
        err = num / den
        assert err <= TOL[cfg.dtype], f"{name} bias={bias}: rel err {err:.3e} over {n} outputs"
        del dinp, out
        torch.cuda.empty_cache()


# --------------------------------------------------------------------------
# transpose_weight: weight[r] stored as (El, H, Kp)
# --------------------------------------------------------------------------

TW_CASES = [
    (2, 2, 4, 96, 256, 512, 0, "fp16"),
    (4, 2, 8, 40, 208, 328, 1, "bf16"),
    (8, 4, 16, 64, 256, 256, 1, "fp16"),
    (2, 2, 4, 6, 12, 10, 0, "bf16"),          # unaligned: not for the TMA kernels
    (2, 2, 4, 40, 130, 70, 1, "fp16"),        # unaligned, several K blocks
    (2, 2, 4, 40, 256, 70, 1, "fp16"),        # H = 70 ragged, but transposed rows are Kp = 128
]


@pytest.mark.parametrize("variant", ["tc", "tc2", "tcr", "tcu", "simt"])
@pytest.mark.parametrize("case", TW_CASES)
def test_transposed_weight(case, variant):
    ep, tp, E, C, M, H, t, dt = case
    cfg = FusedConfig("tw", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=sum(case[:6]) + 5)
    inp = fused_inputs_host(cfg)
    ref = _oracle(cfg, inp)
    dinp = _to_dev(inp)
    wt = [w.transpose(1, 2).contiguous() for w in dinp["w"]]
    ys = bra.bmm_rs_a2a_infer_shape(ep, tp, E, C, M, H, t)["y"]
    out = [torch.full(ys, float("nan"), dtype=dinp["x"][0].dtype, device="cuda")
           for _ in range(cfg.P)]
    aligned = (M // tp) % 8 == 0          # TMA-ready x rows and (Kp-long) weight rows
    if variant in ("tc", "tc2") and not aligned:
        with pytest.raises(bra.BraError):
            bra.bmm_rs_a2a(dinp["x"], wt, dinp["bias"], ep, tp, E, C, M, H, t, out=out,
                           transpose_weight=True, variant=variant)
        return
    bra.bmm_rs_a2a(dinp["x"], wt, dinp["bias"], ep, tp, E, C, M, H, t, out=out,
                   transpose_weight=True, variant=variant)
    torch.cuda.synchronize()
    assert bra.fault_status() == 0
    err = _rel_err(out, ref)
    assert err <= TOL[dt], f"{case} {variant} transposed: rel err {err:.3e}"


def test_transposed_weight_full_size_every_tile():
    cfg = FUSED_CONFIGS["ep8tp2_E64_C256_M4096_H4096_t0_bf16"]
    dinp = fused_inputs_device(cfg)
    wt = [w.transpose(1, 2).contiguous() for w in dinp["w"]]
    ys = bra.bmm_rs_a2a_infer_shape(cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, 0)["y"]
    out = [torch.full(ys, float("nan"), dtype=torch.bfloat16, device="cuda")
           for _ in range(cfg.P)]
    bra.bmm_rs_a2a(dinp["x"], wt, dinp["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, 0,
                   out=out, transpose_weight=True)
    torch.cuda.synchronize()
    assert bra.fault_status() == 0
    for y in out:
        assert not torch.isnan(y).any().item()
    rng = np.random.default_rng(7)
    err = _points_check(cfg, {"x": dinp["x"], "w": wt, "bias": dinp["bias"]}, out,
                        _tile_points(cfg, rng) + _sample_points(cfg, rng, per_rank=4),
                        w_transposed=True)
    assert err <= TOL["bf16"], f"rel err {err:.3e}"


@pytest.mark.parametrize("variant", [None, "tcu"])
@pytest.mark.parametrize("transposed", [False, True])
def test_unaligned_large_every_tile(transposed, variant, monkeypatch):
    """A large shape with 4100-byte token rows and 8200-byte weight rows: the
    row-class TMA kernel (the automatic choice) and the load-staged kernel,
    against the oracle at a point in every output tile."""
    cfg = FUSED_CONFIGS["ep8tp2_E64_C256_M4096_H4096_t0_bf16"].replace(E=16, M=4100, H=4100)
    dinp = fused_inputs_device(cfg)
    w = [u.transpose(1, 2).contiguous() for u in dinp["w"]] if transposed else dinp["w"]
    ys = bra.bmm_rs_a2a_infer_shape(cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, 0)["y"]
    out = [torch.full(ys, float("nan"), dtype=torch.bfloat16, device="cuda")
           for _ in range(cfg.P)]
    monkeypatch.delenv("BRA_FORCE_VARIANT", raising=False)
    assert bra.bmm_rs_a2a_variant(dinp["x"], w, dinp["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C,
                                  cfg.M, cfg.H, 0, out, transpose_weight=transposed) == \
        bra.VARIANT_TCR
    bra.bmm_rs_a2a(dinp["x"], w, dinp["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, 0,
                   out=out, transpose_weight=transposed, variant=variant)
    torch.cuda.synchronize()
    assert bra.fault_status() == 0
    for y in out:
        assert not torch.isnan(y).any().item()
    rng = np.random.default_rng(11)
    err = _points_check(cfg, dinp, out, _tile_points(cfg, rng) + _sample_points(cfg, rng, 4))
    assert err <= TOL["bf16"], f"rel err {err:.3e}"


@pytest.mark.parametrize("variant", [None, "tc", "tc2"])
@pytest.mark.parametrize("case", [
    (2, 2, 4, 64, 256, 24, 0, "fp16"),        # H/tp = 12: output rows of 24 bytes
    (4, 2, 8, 256, 512, 1032, 0, "bf16"),     # H/tp = 516, 256 x 256 pair tiles
    (2, 4, 4, 96, 512, 264, 0, "bf16"),       # H/tp = 66
])
def test_tma_kernels_with_unaligned_output_rows(case, variant, monkeypatch):
    """x and weight rows are TMA-ready, the yShardType-0 output rows are not:
    the TMA kernels store element by element."""
    ep, tp, E, C, M, H, t, dt = case
    for bias in (True, False):
        cfg = FusedConfig("yo", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                          seed=sum(case[:6]) + 31, has_bias=bias)
        inp = fused_inputs_host(cfg)
        dinp = _to_dev(inp)
        if variant is None:
            ys = bra.bmm_rs_a2a_infer_shape(ep, tp, E, C, M, H, t)["y"]
            probe = [torch.empty(ys, dtype=dinp["x"][0].dtype, device="cuda")
                     for _ in range(cfg.P)]
            monkeypatch.delenv("BRA_FORCE_VARIANT", raising=False)
            assert bra.bmm_rs_a2a_variant(dinp["x"], dinp["w"], dinp["bias"], ep, tp, E, C, M,
                                          H, t, probe) in (bra.VARIANT_TC, bra.VARIANT_TC2)
        out = _run(cfg, dinp, variant, monkeypatch)
        err = _rel_err(out, _oracle(cfg, inp))
        assert err <= TOL[dt], f"{case} {variant} bias={bias}: rel err {err:.3e}"


@pytest.mark.parametrize("variant", ["tc", "tc2"])
def test_tma_kernels_with_element_aligned_outputs_and_bias(variant, monkeypatch):
    """16-byte x and weight, but y and bias views start a few elements past a
    16-byte boundary: element-wise epilogue, same results as the oracle."""
    cfg = FusedConfig("yb", ep=4, tp=2, E=8, C=128, M=512, H=768, y_shard_type=1,
                      dtype="fp16", seed=41)
    inp = fused_inputs_host(cfg)
    dinp = _to_dev(inp)
    bias = [_shifted(b, 1 + r % 5) for r, b in enumerate(dinp["bias"])]
    ys = bra.bmm_rs_a2a_infer_shape(cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, 1)["y"]
    outs = [_shifted(torch.full(ys, float("nan"), dtype=torch.float16, device="cuda"),
                     1 + r % 7) for r in range(cfg.P)]
    bra.bmm_rs_a2a(dinp["x"], dinp["w"], bias, cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, 1,
                   out=outs, variant=variant)
    torch.cuda.synchronize()
    assert bra.fault_status() == 0
    assert _rel_err(outs, _oracle(cfg, inp)) <= TOL["fp16"]


def _shifted(t, off):
    """A copy of t whose storage starts `off` elements past an allocation
    (16-byte aligned) start."""
    buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=t.device)
    v = buf[off:off + t.numel()].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("transposed", [False, True])
@pytest.mark.parametrize("M,H", [(272, 264), (130, 70)])
def test_element_aligned_pointers(M, H, transposed, monkeypatch):
    """x, weight and y of every rank start 1..7 elements past a 16-byte
    boundary (a different offset per rank), with 16-byte and with unaligned
    row pitches: the row-class maps start below each row and the rows are
    shifted into place."""
    cfg = FusedConfig("ptr", ep=4, tp=2, E=8, C=96, M=M, H=H, y_shard_type=1, dtype="bf16",
                      seed=M + H)
    inp = fused_inputs_host(cfg)
    ref = _oracle(cfg, inp)
    dinp = _to_dev(inp)
    xs = [_shifted(x, 1 + r % 7) for r, x in enumerate(dinp["x"])]
    w0 = [w.transpose(1, 2).contiguous() for w in dinp["w"]] if transposed else dinp["w"]
    ws = [_shifted(w, 7 - r % 7) for r, w in enumerate(w0)]
    ys = bra.bmm_rs_a2a_infer_shape(cfg.ep, cfg.tp, cfg.E, cfg.C, M, H, 1)["y"]
    outs = [_shifted(torch.full(ys, float("nan"), dtype=torch.bfloat16, device="cuda"), 3)
            for _ in range(cfg.P)]
    monkeypatch.delenv("BRA_FORCE_VARIANT", raising=False)
    for v in (None, "tcu"):
        assert v or bra.bmm_rs_a2a_variant(xs, ws, dinp["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C,
                                           M, H, 1, outs, transpose_weight=transposed) == \
            bra.VARIANT_TCR
        for o in outs:
            o.fill_(float("nan"))
        bra.bmm_rs_a2a(xs, ws, dinp["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C, M, H, 1, out=outs,
                       transpose_weight=transposed, variant=v)
        torch.cuda.synchronize()
        assert bra.fault_status() == 0
        err = _rel_err(outs, ref)
        assert err <= TOL["bf16"], f"M={M} H={H} transposed={transposed} {v}: {err:.3e}"


# --------------------------------------------------------------------------
# The limits the guide's constraints allow (约束说明 / 数据关系与取值范围说明)
# --------------------------------------------------------------------------

MAX_CASES = [
    # ep, tp, E, C, M, H, type, dtype, variants
    (32, 32, 32, 2, 256, 256, 0, "fp16", ("tc", "tcr", "tcu", "simt")),  # P = 1024 virtual ranks
    (32, 32, 32, 32, 256, 256, 1, "bf16", ("tc", "tcr", "tcu")),         # P = 1024, C/tp = 1
    (16, 2, 512, 1, 16, 16, 0, "fp16", ("tc", "tcr", "tcu")),            # E = 512: 32 local experts
    (2, 1, 2, 2, 16, 65535, 0, "bf16", ("tcr", "tcu", "simt")),          # H = 65535 (odd)
    (2, 1, 2, 2, 65535, 16, 1, "fp16", ("tcr", "tcu")),                  # M/tp = 65535 (odd)
]


@pytest.mark.parametrize("case", MAX_CASES)
def test_maximum_sizes(case, monkeypatch):
    ep, tp, E, C, M, H, t, dt, variants = case
    cfg = FusedConfig("max", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=ep + tp + E + C)
    inp = fused_inputs_host(cfg)
    ref = _oracle(cfg, inp)
    dinp = _to_dev(inp)
    for v in variants:
        out = _run(cfg, dinp, v, monkeypatch)
        err = _rel_err(out, ref)
        assert err <= TOL[dt], f"{case[:8]} {v}: rel err {err:.3e}"
        del out
