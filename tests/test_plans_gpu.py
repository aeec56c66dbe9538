"""Prepared calls (Plan): checks once, then only the library call.

A plan gives the same bits as the one-shot function, and a run after the
inputs changed in place (same buffers) sees the new values.
"""
import numpy as np
import pytest
import torch

import bmm_reducescatter_alltoall_gb300 as bra
from workloads import A2AV_CONFIGS, FusedConfig, a2av_index, a2av_inputs, fused_inputs_host

pytestmark = pytest.mark.gpu


def _bits(ts):
    return [t.view(torch.int16 if t.element_size() == 2 else
                   (torch.int32 if t.element_size() == 4 else torch.int8)).cpu() for t in ts]


# TMA kernel, row-class kernel, packed variant (workspace)
@pytest.mark.parametrize("M,H,packed", [(512, 768, False), (514, 774, False), (514, 774, True)])
def test_fused_plan_matches_the_one_shot_call(M, H, packed):
    cfg = FusedConfig("pl", ep=4, tp=2, E=8, C=128, M=M, H=H, y_shard_type=1, dtype="fp16",
                      seed=3)
    inp = fused_inputs_host(cfg)
    d = {k: [u.cuda() for u in v] for k, v in inp.items()}
    args = (cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, cfg.y_shard_type)
    ws = None
    if packed:
        ys = bra.bmm_rs_a2a_infer_shape(*args)["y"]
        probe = [torch.empty(ys, dtype=torch.float16, device="cuda") for _ in range(cfg.P)]
        n = bra.bmm_rs_a2a_workspace_size(d["x"], d["w"], d["bias"], *args, probe)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        assert bra.bmm_rs_a2a_variant(d["x"], d["w"], d["bias"], *args, probe,
                                      workspace=ws) == bra.VARIANT_PACKED
    plan = bra.bmm_rs_a2a_plan(d["x"], d["w"], d["bias"], *args, workspace=ws)
    for step in range(3):
        if step == 2:
            for x in d["x"]:
                x.mul_(-0.5)                       # new values, same buffers
        got = _bits(plan.run())
        ref = _bits(bra.bmm_rs_a2a(d["x"], d["w"], d["bias"], *args, workspace=ws))
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(got, ref)), step
    assert bra.fault_status() == 0


def test_exchange_plans_match_the_one_shot_calls():
    cfg = A2AV_CONFIGS["P32_L64_int8_dirichlet0.3"]
    sc, inputs = a2av_inputs(cfg)
    ins = [torch.from_numpy(a).cuda() for a in inputs]
    idx = [torch.from_numpy(x).cuda()
           for x in a2av_index(sc, [len(a) for a in inputs], "perm", seed=4)]
    scd = torch.from_numpy(sc).cuda()
    mk = lambda: [torch.zeros(int(c), dtype=torch.int8, device="cuda") for c in sc.sum(axis=0)]
    p1 = bra.all_to_all_v_plan(ins, scd, mk(), cfg.L)
    p2 = bra.indexed_all_to_all_v_plan(ins, idx, scd, mk(), cfg.L)
    for step in range(2):
        if step == 1:
            for a in ins:
                a.neg_()
        r1, r2 = p1(), p2()
        o1 = bra.all_to_all_v(ins, scd, mk(), cfg.L)["out"]
        o2 = bra.indexed_all_to_all_v(ins, idx, scd, mk(), cfg.L)["out"]
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(r1["out"], o1))
        assert all(torch.equal(a, b) for a, b in zip(r2["out"], o2))
