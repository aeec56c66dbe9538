"""Seeded synthetic inputs for the fused BMM-RS-Add-A2A op and all_to_all_v.

This module draws random numbers and lays them out in the per-rank shapes the
op's pages fix; it contains none of the method's arithmetic (no matmul, no
reduction, no prefix sum, no permutation).  Both the CPU oracle's tests and the
GPU path's tests, the bench and the smoke check take their inputs from here.

Shapes follow "BatchMatMulReduceScatterAllToAll 原理、shape 约束与 aclnn 两段式调用",
§约束说明 (shape relations):
  yShardType 0: x (E/ep, ep*C, M/tp), weight (E/ep, M/tp, H), bias (E/ep, 1, H/tp)
  yShardType 1: x (E/ep, ep*tp*C/tp, M/tp), weight (E/ep, M/tp, H), bias (E/ep, 1, H)
Bias dtype follows §参数说明: fp16 for fp16 x, fp32 for bf16 x.

Recipes (one generator per case, draws in this order):
  * fused, host:   numpy.random.default_rng(seed); every x_r for r = 0..P-1,
    then every weight_r, then every bias_r; each drawn as float32 standard
    normals times the stated std, then cast to the storage dtype (fp16 via
    numpy, bf16 via torch; both round to nearest even).
  * fused, device: torch.Generator on the device seeded with `seed`, same
    order, torch.randn in float32 times std, then cast.  Used for the large
    workloads (8.6 GB of inputs), which the host would take minutes to draw.
  * all_to_all_v: numpy.random.default_rng(seed); first the P x P count
    matrix, then each rank's payload in rank order.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass
from typing import List, Optional

import numpy as np

__all__ = [
    "FusedConfig", "A2AVConfig", "FUSED_CONFIGS", "A2AV_CONFIGS", "a2av_index",
    "fused_shapes", "fused_inputs_host", "fused_inputs_device",
    "a2av_counts", "a2av_inputs",
]


@dataclass(frozen=True)
class FusedConfig:
    """One fused BMM-RS-Add-A2A workload; P = ep * tp virtual ranks."""
    name: str
    ep: int
    tp: int
    E: int
    C: int
    M: int
    H: int
    y_shard_type: int
    dtype: str            # "fp16" | "bf16"
    seed: int
    x_std: float = 1.0
    w_std: float = 1.0
    bias_std: float = 1.0
    has_bias: bool = True

    @property
    def P(self) -> int:
        return self.ep * self.tp

    @property
    def flops(self) -> int:
        # 2 * E * (ep*C) * M * H multiply-adds over the whole job.
        return 2 * self.E * self.ep * self.C * self.M * self.H

    def replace(self, **kw) -> "FusedConfig":
        return dataclasses.replace(self, **kw)


@dataclass(frozen=True)
class A2AVConfig:
    """One all_to_all_v workload over P virtual ranks with core_num L."""
    name: str
    P: int
    L: int
    dtype: str            # "fp32" | "int8"
    seed: int
    counts: str           # "uniform" | "dirichlet"
    count_max: int = 4096          # uniform: counts in [0, count_max]
    alpha: float = 0.3             # dirichlet concentration
    scale: int = 1 << 21           # dirichlet: counts = rint(scale * w_ij)

    def replace(self, **kw) -> "A2AVConfig":
        return dataclasses.replace(self, **kw)


FUSED_CONFIGS = {
    # 8-rank example of the CANN guide (EP4 x TP2, C-sharded), N(0,1) values.
    "ep4tp2_E16_C12_M12_H4_t1_fp16": FusedConfig(
        "ep4tp2_E16_C12_M12_H4_t1_fp16", ep=4, tp=2, E=16, C=12, M=12, H=4,
        y_shard_type=1, dtype="fp16", seed=0),
    "ep8tp2_E64_C256_M4096_H4096_t0_bf16": FusedConfig(
        "ep8tp2_E64_C256_M4096_H4096_t0_bf16", ep=8, tp=2, E=64, C=256,
        M=4096, H=4096, y_shard_type=0, dtype="bf16", seed=2,
        x_std=0.02, w_std=0.02, bias_std=1.0),
    "ep8tp4_E64_C512_M8192_H4096_t1_fp16": FusedConfig(
        "ep8tp4_E64_C512_M8192_H4096_t1_fp16", ep=8, tp=4, E=64, C=512,
        M=8192, H=4096, y_shard_type=1, dtype="fp16", seed=4,
        x_std=0.02, w_std=0.02, bias_std=1.0),
    # Profiling size of the bf16 workload: the same per-expert GEMMs, one
    # local expert per rank (E = ep), 1/8 of the FLOPs, 0.5 GB on the device.
    "ep8tp2_E8_C256_M4096_H4096_t0_bf16": FusedConfig(
        "ep8tp2_E8_C256_M4096_H4096_t0_bf16", ep=8, tp=2, E=8, C=256,
        M=4096, H=4096, y_shard_type=0, dtype="bf16", seed=2,
        x_std=0.02, w_std=0.02, bias_std=1.0),
    # The bf16 profiling size with 4100-byte token rows and 8200-byte weight
    # rows (M/tp = H/tp = 2050): no TMA descriptor of the whole matrices fits;
    # the row-class TMA kernel runs.
    # Decode-like token counts at profiling size: C = 16 (128 token rows per
    # group), one local expert per rank; the weights (0.54 GB) dominate the
    # bytes, and the one-CTA kernel streams them.
    "ep8tp4_E8_C16_M8192_H4096_t1_fp16": FusedConfig(
        "ep8tp4_E8_C16_M8192_H4096_t1_fp16", ep=8, tp=4, E=8, C=16,
        M=8192, H=4096, y_shard_type=1, dtype="fp16", seed=4,
        x_std=0.02, w_std=0.02, bias_std=1.0),
    "ep8tp2_E8_C256_M4100_H4100_t0_bf16": FusedConfig(
        "ep8tp2_E8_C256_M4100_H4100_t0_bf16", ep=8, tp=2, E=8, C=256,
        M=4100, H=4100, y_shard_type=0, dtype="bf16", seed=2,
        x_std=0.02, w_std=0.02, bias_std=1.0),
    # Profiling size of the workload above: the same per-expert GEMMs, one
    # local expert per rank (E = ep), 1/8 of the FLOPs, 1.3 GB on the device.
    "ep8tp4_E8_C512_M8192_H4096_t1_fp16": FusedConfig(
        "ep8tp4_E8_C512_M8192_H4096_t1_fp16", ep=8, tp=4, E=8, C=512,
        M=8192, H=4096, y_shard_type=1, dtype="fp16", seed=4,
        x_std=0.02, w_std=0.02, bias_std=1.0),
}

A2AV_CONFIGS = {
    "P8_L10_fp32_uniform4096": A2AVConfig(
        "P8_L10_fp32_uniform4096", P=8, L=10, dtype="fp32", seed=1,
        counts="uniform", count_max=4096),
    "P32_L64_int8_dirichlet0.3": A2AVConfig(
        "P32_L64_int8_dirichlet0.3", P=32, L=64, dtype="int8", seed=3,
        counts="dirichlet", alpha=0.3, scale=1 << 21),
}


def fused_shapes(cfg: FusedConfig, bias_ndim: int = 3) -> dict:
    """Per-rank tensor shapes as the CANN guide's §约束说明 lists them."""
    El = cfg.E // cfg.ep
    Kp = cfg.M // cfg.tp
    if cfg.y_shard_type == 0:
        x = (El, cfg.ep * cfg.C, Kp)
        bias_last = cfg.H // cfg.tp
        y = (cfg.E, cfg.C, cfg.H // cfg.tp)
    else:
        x = (El, cfg.ep * cfg.tp * (cfg.C // cfg.tp), Kp)
        bias_last = cfg.H
        y = (cfg.E, cfg.C // cfg.tp, cfg.H)
    bias = (El, 1, bias_last) if bias_ndim == 3 else (El, bias_last)
    return {"x": x, "w": (El, Kp, cfg.H), "bias": bias, "y": y}


def _torch():
    import torch
    return torch


def _dtypes(cfg: FusedConfig):
    torch = _torch()
    if cfg.dtype == "fp16":
        return torch.float16, torch.float16
    if cfg.dtype == "bf16":
        return torch.bfloat16, torch.float32
    raise ValueError(f"fused dtype must be fp16 or bf16, got {cfg.dtype}")


def fused_inputs_host(cfg: FusedConfig, bias_ndim: int = 3) -> dict:
    """Host (CPU torch) tensors: lists x[P], w[P], bias[P] (or None)."""
    torch = _torch()
    xdt, bdt = _dtypes(cfg)
    sh = fused_shapes(cfg, bias_ndim)
    rng = np.random.default_rng(cfg.seed)

    def draw(shape, std, dt):
        a = rng.standard_normal(shape, dtype=np.float32) * np.float32(std)
        if dt == torch.float16:
            return torch.from_numpy(a.astype(np.float16))
        return torch.from_numpy(a).to(dt)

    x = [draw(sh["x"], cfg.x_std, xdt) for _ in range(cfg.P)]
    w = [draw(sh["w"], cfg.w_std, xdt) for _ in range(cfg.P)]
    bias: Optional[List] = None
    if cfg.has_bias:
        bias = [draw(sh["bias"], cfg.bias_std, bdt) for _ in range(cfg.P)]
    return {"x": x, "w": w, "bias": bias}


def fused_inputs_device(cfg: FusedConfig, device="cuda", bias_ndim: int = 3) -> dict:
    """Device tensors drawn by torch's generator on `device` (seeded)."""
    torch = _torch()
    xdt, bdt = _dtypes(cfg)
    sh = fused_shapes(cfg, bias_ndim)
    g = torch.Generator(device=device)
    g.manual_seed(cfg.seed)

    def draw(shape, std, dt):
        a = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        a.mul_(std)
        return a.to(dt)

    x = [draw(sh["x"], cfg.x_std, xdt) for _ in range(cfg.P)]
    w = [draw(sh["w"], cfg.w_std, xdt) for _ in range(cfg.P)]
    bias = None
    if cfg.has_bias:
        bias = [draw(sh["bias"], cfg.bias_std, bdt) for _ in range(cfg.P)]
    return {"x": x, "w": w, "bias": bias}


def a2av_counts(cfg: A2AVConfig, rng: Optional[np.random.Generator] = None) -> np.ndarray:
    """P x P int64 send-count matrix (row i = what rank i sends to each j)."""
    if rng is None:
        rng = np.random.default_rng(cfg.seed)
    P = cfg.P
    if cfg.counts == "uniform":
        return rng.integers(0, cfg.count_max + 1, size=(P, P), dtype=np.int64)
    if cfg.counts == "dirichlet":
        w = rng.dirichlet(np.full(P, cfg.alpha), size=P)
        return np.rint(w * float(cfg.scale)).astype(np.int64)
    raise ValueError(cfg.counts)


def a2av_inputs(cfg: A2AVConfig, extra: int = 0):
    """(counts, inputs): inputs[i] holds rank i's payload, one value per
    element it sends (its row total), plus `extra` trailing values."""
    rng = np.random.default_rng(cfg.seed)
    counts = a2av_counts(cfg, rng)
    inputs = []
    for i in range(cfg.P):
        n = int(counts[i].sum()) + extra
        if cfg.dtype == "fp32":
            inputs.append(rng.standard_normal(n, dtype=np.float32))
        elif cfg.dtype == "int8":
            inputs.append(rng.integers(-128, 128, size=n, dtype=np.int8))
        else:
            raise ValueError(cfg.dtype)
    return counts, inputs


def a2av_index(counts: np.ndarray, in_lens, kind: str = "perm", seed: int = 0):
    """Index arrays for the indexed exchange: index[i] has one int64 entry per
    element rank i sends (its row total).  kind "perm": a permutation of
    rank i's input positions (needs in_lens[i] == the row total); "random":
    uniform positions in [0, in_lens[i]), repeats allowed; "identity": 0, 1, ..."""
    out = []
    for i in range(len(in_lens)):
        n = int(np.asarray(counts)[i].sum())
        rng = np.random.default_rng([seed, i])
        if kind == "perm":
            assert int(in_lens[i]) == n
            out.append(rng.permutation(n).astype(np.int64))
        elif kind == "random":
            out.append(rng.integers(0, max(int(in_lens[i]), 1), size=n, dtype=np.int64))
        elif kind == "identity":
            out.append(np.arange(n, dtype=np.int64))
        else:
            raise ValueError(kind)
    return out

