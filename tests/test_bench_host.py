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
