"""The calls are stateless: concurrent calls on different streams, and calls
captured in a CUDA graph, give the same bits as eager calls on one stream.

Covers the claim of the C header that calls with disjoint outputs may
overlap on different streams, and the CUDA-graph replay the bench's size
sweep relies on.  The packed variant (repack into a caller workspace, then
the TMA kernel) is among the calls; concurrent calls each have their own
workspace.
"""
import numpy as np
import pytest
import torch

import bmm_reducescatter_alltoall_gb300 as bra
from workloads import A2AV_CONFIGS, FusedConfig, a2av_index, a2av_inputs, fused_inputs_host

pytestmark = pytest.mark.gpu


def _fused_case(seed, t=1, dt="fp16", M=512, H=768):
    cfg = FusedConfig("s", ep=4, tp=2, E=8, C=128, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=seed)
    inp = fused_inputs_host(cfg)
    d = {k: (None if v is None else [u.cuda() for u in v]) for k, v in inp.items()}
    ys = bra.bmm_rs_a2a_infer_shape(cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, t)["y"]
    mk = lambda: [torch.zeros(ys, dtype=d["x"][0].dtype, device="cuda") for _ in range(cfg.P)]
    return cfg, d, mk


def _call(cfg, d, out, stream=None, ws=None):
    bra.bmm_rs_a2a(d["x"], d["w"], d["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H,
                   cfg.y_shard_type, out=out, stream=stream, workspace=ws)


def _workspace(cfg, d, mk):
    n = bra.bmm_rs_a2a_workspace_size(d["x"], d["w"], d["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C,
                                      cfg.M, cfg.H, cfg.y_shard_type, mk())
    assert n > 0
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def _a2av_case():
    cfg = A2AV_CONFIGS["P8_L10_fp32_uniform4096"]
    sc, inputs = a2av_inputs(cfg)
    ins = [torch.from_numpy(a).cuda() for a in inputs]
    scd = torch.from_numpy(sc).cuda()
    mk = lambda: [torch.zeros(int(c), dtype=torch.float32, device="cuda") for c in sc.sum(axis=0)]
    return cfg, ins, scd, mk


def _indexed_case():
    cfg = A2AV_CONFIGS["P8_L10_fp32_uniform4096"]
    sc, inputs = a2av_inputs(cfg, extra=100)
    idx = [torch.from_numpy(x).cuda()
           for x in a2av_index(sc, [len(a) for a in inputs], "random", seed=2)]
    ins = [torch.from_numpy(a).cuda() for a in inputs]
    scd = torch.from_numpy(sc).cuda()
    mk = lambda: [torch.zeros(int(c), dtype=torch.float32, device="cuda") for c in sc.sum(axis=0)]
    return cfg, ins, idx, scd, mk


def _same_bits(a, b):
    return all(torch.equal(x.view(torch.int16) if x.dtype != torch.float32 else x.view(torch.int32),
                           y.view(torch.int16) if y.dtype != torch.float32 else y.view(torch.int32))
               for x, y in zip(a, b))


def test_concurrent_calls_on_three_streams():
    c1, d1, mk1 = _fused_case(1, t=1, dt="fp16")
    c2, d2, mk2 = _fused_case(2, t=0, dt="bf16")
    c3, d3, mk3 = _fused_case(4, t=1, dt="bf16", M=514, H=774)   # Kp = 257: row-class kernel
    assert bra.bmm_rs_a2a_variant(d3["x"], d3["w"], d3["bias"], c3.ep, c3.tp, c3.E, c3.C, c3.M,
                                  c3.H, 1, mk3()) == bra.VARIANT_TCR
    c4, d4, mk4 = _fused_case(6, t=0, dt="fp16", M=514, H=778)   # packed with a workspace
    ws4 = _workspace(c4, d4, mk4)
    ca, ins, scd, mka = _a2av_case()
    ci, iins, iidx, iscd, mki = _indexed_case()
    ref1, ref2, ref3, ref4, refa, refi = mk1(), mk2(), mk3(), mk4(), mka(), mki()
    _call(c1, d1, ref1)
    _call(c2, d2, ref2)
    _call(c3, d3, ref3)
    _call(c4, d4, ref4, ws=ws4)
    bra.all_to_all_v(ins, scd, refa, ca.L)
    bra.indexed_all_to_all_v(iins, iidx, iscd, refi, ci.L)
    torch.cuda.synchronize()
    s1, s2, s3 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        o1, o2, o3, o4, oa, oi = mk1(), mk2(), mk3(), mk4(), mka(), mki()
        torch.cuda.synchronize()
        _call(c1, d1, o1, stream=s1)
        _call(c2, d2, o2, stream=s2)
        _call(c3, d3, o3, stream=s3)
        _call(c4, d4, o4, stream=s2, ws=ws4)
        bra.all_to_all_v(ins, scd, oa, ca.L, stream=s2)
        bra.indexed_all_to_all_v(iins, iidx, iscd, oi, ci.L, stream=s1)
        torch.cuda.synchronize()
        assert _same_bits(o1, ref1) and _same_bits(o2, ref2) and _same_bits(o3, ref3)
        assert _same_bits(o4, ref4)
        assert _same_bits(oa, refa) and _same_bits(oi, refi)
    assert bra.fault_status() == 0


def test_step_captured_in_a_cuda_graph():
    c1, d1, mk1 = _fused_case(3, t=1, dt="fp16")
    c3, d3, mk3 = _fused_case(5, t=0, dt="fp16", M=514, H=774)   # row-class kernel
    ws3 = _workspace(c3, d3, mk3)                                 # and packed
    ca, ins, scd, mka = _a2av_case()
    ci, iins, iidx, iscd, mki = _indexed_case()
    ref1, ref3, refa, refi = mk1(), mk3(), mka(), mki()
    _call(c1, d1, ref1)
    _call(c3, d3, ref3)
    bra.all_to_all_v(ins, scd, refa, ca.L)
    bra.indexed_all_to_all_v(iins, iidx, iscd, refi, ci.L)
    torch.cuda.synchronize()
    o1, o3, o3p, oa, oi = mk1(), mk3(), mk3(), mka(), mki()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # warm the library's per-device set-up
        _call(c1, d1, o1)
        _call(c3, d3, o3)
        _call(c3, d3, o3p, ws=ws3)
        bra.all_to_all_v(ins, scd, oa, ca.L)
        bra.indexed_all_to_all_v(iins, iidx, iscd, oi, ci.L)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref3p = [t_.clone() for t_ in o3p]
    for t_ in o1 + o3 + o3p + oa + oi:
        t_.zero_()
    ws3.fill_(0x5A)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _call(c1, d1, o1)
        _call(c3, d3, o3)
        _call(c3, d3, o3p, ws=ws3)
        bra.all_to_all_v(ins, scd, oa, ca.L)
        bra.indexed_all_to_all_v(iins, iidx, iscd, oi, ci.L)
    for _ in range(2):
        for t_ in o1 + o3 + o3p + oa + oi:
            t_.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert _same_bits(o1, ref1) and _same_bits(o3, ref3) and _same_bits(oa, refa)
        assert _same_bits(oi, refi) and _same_bits(o3p, ref3p)
        # the packed variant agrees with the row-class kernel to the output rounding
        for a, b in zip(o3p, ref3):
            assert torch.allclose(a.float(), b.float(), rtol=2e-3, atol=2e-3 * b.float().abs().max().item())
    assert bra.fault_status() == 0
