"""Failure detection on the GPU without a fault: a bounded wait runs out.

Each wait helper (the one every mbarrier wait of all_to_all_v, of the
tensor-core fused kernels, or the cluster-scope wait of the row-class
kernel's MMA issuer goes through) is run on a barrier phase that nothing
completes.  The wait gives up after its limit
(about 2 s / 4 s), the kernel reports BRA_ERR_TIMEOUT in its status word and
in the watchdog word the host reads, and returns; nothing traps, and the
context stays usable, which the exact exchange run afterwards checks.
"""
import numpy as np
import pytest
import torch

import bmm_reducescatter_alltoall_gb300 as bra
from oracle import a2av as oa
from workloads import A2AV_CONFIGS, a2av_inputs

pytestmark = pytest.mark.gpu


def _exchange_is_exact():
    cfg = A2AV_CONFIGS["P8_L10_fp32_uniform4096"]
    sc, inputs = a2av_inputs(cfg)
    ins = [torch.from_numpy(a).cuda() for a in inputs]
    outs = [torch.zeros(int(c), dtype=torch.float32, device="cuda") for c in sc.sum(axis=0)]
    bra.all_to_all_v(ins, torch.from_numpy(sc).cuda(), outs, cfg.L)
    torch.cuda.synchronize()
    ref = oa.all_to_all_v(inputs, sc, [np.zeros(int(c), np.float32) for c in sc.sum(axis=0)])
    return all(np.array_equal(o.cpu().numpy().view(np.uint32), r.view(np.uint32))
               for o, r in zip(outs, ref["out"]))


@pytest.mark.parametrize("which", ["a2av", "tc", "tc_cluster"])
def test_bounded_wait_runs_out_and_reports(which):
    bra.fault_status(clear=True)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    bra.wait_selftest(which, status)
    torch.cuda.synchronize()
    assert int(status.item()) == bra.ERR_TIMEOUT
    assert bra.fault_status() == bra.ERR_TIMEOUT
    bra.fault_status(clear=True)
    assert bra.fault_status() == 0
    assert _exchange_is_exact()
    assert bra.fault_status() == 0


def test_fused_status_word_is_the_calls_own():
    """A bounded wait that runs out on one stream sets the device's watchdog
    word, which every call shares, but not the status word of a fused call
    running meanwhile on another stream: that word is set to 0 before the
    call's kernels and stays 0, and the call's output matches the oracle."""
    from oracle import fused as of
    from workloads import FUSED_CONFIGS, fused_inputs_host

    bra.fault_status(clear=True)
    cfg = FUSED_CONFIGS["ep4tp2_E16_C12_M12_H4_t1_fp16"].replace(name="st", C=128, M=256, H=256)
    inp = fused_inputs_host(cfg)
    dev = {k: [t.cuda() for t in v] for k, v in inp.items()}
    probe_status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    call_status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    bra.wait_selftest("tc", probe_status, stream=s1)
    out = bra.bmm_rs_a2a(dev["x"], dev["w"], dev["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M,
                         cfg.H, cfg.y_shard_type, stream=s2, status=call_status)
    s2.synchronize()
    assert int(call_status.item()) == 0      # done while the probe still waits
    torch.cuda.synchronize()
    assert int(probe_status.item()) == bra.ERR_TIMEOUT
    assert bra.fault_status() == bra.ERR_TIMEOUT
    assert int(call_status.item()) == 0
    ref = of.bmm_rs_a2a(inp["x"], inp["w"], inp["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M,
                        cfg.H, cfg.y_shard_type, cfg.dtype)
    g = np.concatenate([o.float().cpu().numpy().ravel() for o in out]).astype(np.float64)
    r = np.concatenate([a.ravel() for a in ref])
    assert np.max(np.abs(g - r)) / np.max(np.abs(r)) <= 2e-3
    bra.fault_status(clear=True)
    assert bra.fault_status() == 0
