"""The full-size parity checks' point selection, run on the CPU.

The GPU tests compare the fused kernels with the oracle at one point inside
every 128 x 256 tile of every sender group's product.  Here the selection is
checked against the oracle itself on small problems: each tile of each group
gets exactly one point, each point is where the oracle's receiver view says
that product entry goes, the checker reports zero error on the oracle's own
outputs (with the weight in either layout), and a wrong value planted at
one of the points is caught.
"""
import numpy as np
import pytest
import torch

from oracle import fused as of
from test_fused_gpu import _points_check, _sample_points, _tile_points
from workloads import FusedConfig, fused_inputs_host

CASES = [(4, 2, 8, 200, 24, 600, 1, "fp16"), (2, 4, 4, 96, 32, 520, 0, "bf16"),
         (2, 2, 4, 130, 16, 300, 0, "fp16"), (1, 1, 2, 300, 8, 257, 1, "bf16")]


@pytest.mark.parametrize("case", CASES)
def test_one_point_per_tile_aimed_at_its_product_entry(case):
    ep, tp, E, C, M, H, t, dt = case
    cfg = FusedConfig("h", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt, seed=3)
    pts = _tile_points(cfg, np.random.default_rng(1))
    El, rows = E // ep, ep * C
    seen = {}
    for d, i, c, h, zrow, zcol in pts:
        src = of.y_source(ep, tp, E, C, H, t, d, i, c, h)
        assert (src["zrow"], src["zcol"]) == (zrow, zcol)
        key = (src["s"] * El + src["e"], zrow // 128, zcol // 256)
        assert key not in seen
        seen[key] = 1
    assert len(seen) == ep * El * (-(-rows // 128)) * (-(-H // 256))


@pytest.mark.parametrize("case", CASES)
def test_checker_is_zero_on_the_oracle_and_catches_a_planted_error(case):
    ep, tp, E, C, M, H, t, dt = case
    cfg = FusedConfig("h", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt, seed=3)
    inp = fused_inputs_host(cfg)
    ref = of.bmm_rs_a2a(inp["x"], inp["w"], inp["bias"], ep, tp, E, C, M, H, t, dt)
    tdt = torch.float16 if dt == "fp16" else torch.bfloat16
    out = [torch.from_numpy(r).to(tdt) for r in ref]
    rng = np.random.default_rng(2)
    pts = _tile_points(cfg, rng) + _sample_points(cfg, rng, 4)
    assert _points_check(cfg, inp, out, pts) == 0.0
    wt = {"x": inp["x"], "w": [w.transpose(1, 2).contiguous() for w in inp["w"]],
          "bias": inp["bias"]}
    assert _points_check(cfg, wt, out, pts, w_transposed=True) == 0.0
    d, i, c, h = pts[len(pts) // 2][:4]
    out[d][i, c, h] += 1.0
    assert _points_check(cfg, inp, out, pts) > 1e-2
