"""The bench's unfused context leg computes the same op as the oracle."""
import numpy as np
import pytest
import torch

import bench
from oracle import fused as of
from workloads import FUSED_CONFIGS, FusedConfig, fused_inputs_host


@pytest.mark.parametrize("cfg", [
    FUSED_CONFIGS["ep4tp2_E16_C12_M12_H4_t1_fp16"],
    FUSED_CONFIGS["ep4tp2_E16_C12_M12_H4_t1_fp16"].replace(y_shard_type=0),
    FusedConfig("b", ep=2, tp=2, E=4, C=8, M=16, H=8, y_shard_type=0, dtype="bf16", seed=5),
    FusedConfig("nb", ep=2, tp=4, E=2, C=8, M=32, H=8, y_shard_type=1, dtype="fp16", seed=6,
                has_bias=False),
])
def test_unfused_reference_matches_oracle(cfg):
    inp = fused_inputs_host(cfg)
    f32 = lambda v: None if v is None else [t.float() for t in v]
    ys = of.infer_shapes(cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, cfg.y_shard_type)["y"]
    out = [torch.zeros(ys) for _ in range(cfg.P)]
    bench.unfused_torch(cfg, f32(inp["x"]), f32(inp["w"]), f32(inp["bias"]), out)
    ref = of.bmm_rs_a2a(inp["x"], inp["w"], inp["bias"], cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M,
                        cfg.H, cfg.y_shard_type, cfg.dtype)
    err = max(float(np.max(np.abs(o.numpy() - r))) for o, r in zip(out, ref))
    err /= max(float(np.max(np.abs(r))) for r in ref)
    assert err <= (2e-3 if cfg.dtype == "fp16" else 1e-2)


def test_arguments_and_defaults():
    """The driver's contract: no flags give N = 1, K/W within minutes, the
    headline workloads; --workspace and the profiling switches parse."""
    a = bench._args([])
    assert (a.gpus, a.warmup, a.impl, a.fused, a.a2av) == (1, 3, "ours", bench.FUSED_NAME,
                                                          bench.A2AV_NAME)
    assert a.steps >= 1 and a.warmup >= 3 and not a.workspace
    b = bench._args(["--workspace", "--fused", "ep8tp2_E8_C256_M4100_H4100_t0_bf16",
                     "--steps", "3", "--e2e-steps", "0", "--indexed-calls", "0"])
    assert b.workspace and b.steps == 3 and b.e2e_steps == 0 and b.indexed_calls == 0
    assert b.fused in FUSED_CONFIGS


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def test_clock_sampler_reads_the_timed_window_and_reasons():
    """The clock record of the bench line: the median SM clock, the maximum
    clock and power, and the active throttle reasons of the samples inside
    the timed window only (fields as nvidia-smi's CSV gives them)."""
    s = bench.ClockSampler(0)
    s.proc = _FakeProc()
    row = lambda mhz, pw, cap, thermal: [
        "0", str(mhz), "2070", str(pw), "0x4", "Not Active",
        "Active" if thermal else "Not Active", "Not Active", "Active" if cap else "Not Active"]
    s.rows = [(0.5, row(2070, 300.0, False, True)),           # before the window
              (1.0, row(1300, 1390.5, True, False)),
              (1.5, row(1320, 1401.0, True, False)),
              (2.0, row(1310, 1395.0, False, False)),
              (3.5, row(2070, 200.0, False, True))]           # after it
    s.mark(0.9, 2.1)
    rec = s.stop()
    assert rec["sm_mhz"] == 1310 and rec["sm_max_mhz"] == 2070
    assert rec["power_w_max"] == 1401.0 and rec["samples"] == 3
    assert rec["reasons"] == ["sw_power_cap"]
    s2 = bench.ClockSampler(0)
    s2.proc = _FakeProc()
    s2.rows = [(1.0, row(1800, 900.0, False, True))]
    s2.mark(0.5, 1.5)
    assert s2.stop()["reasons"] == ["hw_thermal_slowdown"]
