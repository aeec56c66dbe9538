"""Randomised and repeated runs, to catch what fixed cases can miss.

* Random shapes with rows of any alignment (both shard types, bias or not,
  weight stored either way, pointers offset by a few elements) run on the
  automatic kernel choice, half of them given a workspace (the packed
  variant where the rows lack a 16-byte pitch), and are compared with the
  oracle.
* Every kernel runs the same inputs several times: each output element has
  one fixed accumulation order, so the results must be bit-identical call to
  call.  A synchronisation slip between the roles of a kernel (a stage read
  before it is complete, or overwritten while still in use) would show here.
"""
import numpy as np
import pytest
import torch

import bmm_reducescatter_alltoall_gb300 as bra
from oracle import fused as of
from workloads import A2AV_CONFIGS, FusedConfig, a2av_index, a2av_inputs, fused_inputs_host

pytestmark = pytest.mark.gpu

TOL = {"fp16": 2e-3, "bf16": 1e-2}


def _shifted(t, off):
    buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=t.device)
    v = buf[off:off + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def _random_config(rng, k):
    ep = int(rng.choice([1, 2, 4]))
    tp = int(rng.choice([1, 2, 4]))
    El = int(rng.integers(1, 3))
    if El * ep < 2:                                   # E = El * ep must be at least 2
        El = 2
    t = int(rng.integers(0, 2))
    C = tp * int(rng.integers(1, 40)) if t == 1 else int(rng.integers(1, 150))
    Kp = int(rng.integers(1, 300))
    H = tp * int(rng.integers(1, 120)) if t == 0 else int(rng.integers(1, 400))
    dt = "fp16" if rng.random() < 0.5 else "bf16"
    return FusedConfig(f"fz{k}", ep=ep, tp=tp, E=El * ep, C=C, M=Kp * tp, H=H, y_shard_type=t,
                       dtype=dt, seed=1000 + k, has_bias=bool(rng.random() < 0.7))


@pytest.mark.parametrize("k", range(24))
def test_random_shapes_match_the_oracle(k):
    rng = np.random.default_rng(500 + k)
    cfg = _random_config(rng, k)
    transposed = bool(rng.random() < 0.4)
    inp = fused_inputs_host(cfg)
    ref = of.bmm_rs_a2a(inp["x"], inp["w"], inp["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M,
                        cfg.H, cfg.y_shard_type, cfg.dtype)
    offs = rng.integers(0, 8, size=2 * cfg.P)
    xs = [_shifted(x.cuda(), int(offs[r])) for r, x in enumerate(inp["x"])]
    w0 = [w.cuda() for w in inp["w"]]
    if transposed:
        w0 = [w.transpose(1, 2).contiguous() for w in w0]
    ws = [_shifted(w, int(offs[cfg.P + r])) for r, w in enumerate(w0)]
    bias = None if inp["bias"] is None else [b.cuda() for b in inp["bias"]]
    ys = bra.bmm_rs_a2a_infer_shape(cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H,
                                    cfg.y_shard_type)["y"]
    out = [torch.full(ys, float("nan"), dtype=xs[0].dtype, device="cuda") for _ in range(cfg.P)]
    workspace = None
    if rng.random() < 0.5:                        # the packed variant where it applies
        n = bra.bmm_rs_a2a_workspace_size(xs, ws, bias, cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M,
                                          cfg.H, cfg.y_shard_type, out,
                                          transpose_weight=transposed)
        if n > 0:
            workspace = torch.full((n,), 0xA5, dtype=torch.uint8, device="cuda")
    bra.bmm_rs_a2a(xs, ws, bias, cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, cfg.y_shard_type,
                   out=out, transpose_weight=transposed, workspace=workspace)
    torch.cuda.synchronize()
    assert bra.fault_status() == 0
    g = np.concatenate([o.float().cpu().numpy().ravel() for o in out]).astype(np.float64)
    r = np.concatenate([a.ravel() for a in ref])
    assert np.isfinite(g).all(), "an output element was not written"
    err = float(np.max(np.abs(g - r)) / max(np.max(np.abs(r)), 1e-30))
    assert err <= TOL[cfg.dtype], f"{cfg} transposed={transposed}: rel err {err:.3e}"


def _fused_repeat(variant, M, H, t, dt, monkeypatch, calls=5):
    cfg = FusedConfig("rep", ep=4, tp=2, E=8, C=160, M=M, H=H, y_shard_type=t, dtype=dt, seed=7)
    inp = fused_inputs_host(cfg)
    d = {k: (None if v is None else [u.cuda() for u in v]) for k, v in inp.items()}
    ys = bra.bmm_rs_a2a_infer_shape(cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, t)["y"]
    monkeypatch.setenv("BRA_FORCE_VARIANT", variant)
    outs = []
    for _ in range(calls):
        o = [torch.zeros(ys, dtype=d["x"][0].dtype, device="cuda") for _ in range(cfg.P)]
        bra.bmm_rs_a2a(d["x"], d["w"], d["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, t,
                       out=o)
        outs.append(o)
    torch.cuda.synchronize()
    assert bra.fault_status() == 0
    first = [x.view(torch.int16).cpu() for x in outs[0]]
    for o in outs[1:]:
        for a, b in zip(first, o):
            assert torch.equal(a, b.view(torch.int16).cpu()), f"{variant}: results differ"


@pytest.mark.parametrize("variant,M,H", [("tc2", 1024, 512), ("tc", 1024, 512),
                                         ("tcr", 1026, 518), ("tcu", 1026, 518),
                                         ("tc2", 1024, 520)])   # H/tp = 260: element stores
@pytest.mark.parametrize("t", [0, 1])
def test_repeated_fused_calls_are_bit_identical(variant, M, H, t, monkeypatch):
    _fused_repeat(variant, M, H, t, "bf16" if t == 0 else "fp16", monkeypatch)


def test_repeated_exchanges_are_bit_identical():
    cfg = A2AV_CONFIGS["P32_L64_int8_dirichlet0.3"]
    sc, inputs = a2av_inputs(cfg)
    ins = [torch.from_numpy(a).cuda() for a in inputs]
    idx = [torch.from_numpy(x).cuda()
           for x in a2av_index(sc, [len(a) for a in inputs], "perm", seed=2)]
    scd = torch.from_numpy(sc).cuda()
    cols = sc.sum(axis=0)
    res = {"plain": [], "indexed": []}
    for _ in range(4):
        o = [torch.zeros(int(c), dtype=torch.int8, device="cuda") for c in cols]
        bra.all_to_all_v(ins, scd, o, cfg.L)
        res["plain"].append(o)
        o = [torch.zeros(int(c), dtype=torch.int8, device="cuda") for c in cols]
        bra.indexed_all_to_all_v(ins, idx, scd, o, cfg.L)
        res["indexed"].append(o)
    torch.cuda.synchronize()
    for k, runs in res.items():
        for o in runs[1:]:
            assert all(torch.equal(a, b) for a, b in zip(runs[0], o)), k
