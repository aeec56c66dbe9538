"""bmm_rs_a2a_noalloc: the packed variant with the library's own scratch array.

Some callers cannot allocate device memory for a workspace (a plugin whose
host program owns all device memory, or a path where cudaMalloc's possible
device synchronisation is not allowed).  bmm_rs_a2a_noalloc serves them from
a fixed device array inside the library.  These tests call it through the C
ABI and compare its outputs with those of the existing entry point,
bmm_rs_a2a_ex with the packed variant and a torch-allocated workspace, on
two calls in a row with different inputs (the second call finds the first
call's copies in the shared array).

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import bmm_reducescatter_alltoall_gb300 as bra
from test_abi_host import Fake
from workloads import FusedConfig, fused_inputs_host

TOL = {"fp16": 2e-3, "bf16": 1e-2}
UNSUPPORTED, NULLPTR = 161003, 161001

CASES = [
    # ep, tp, E, C, M, H, yShardType, dtype, weight transposed
    (4, 2, 16, 12, 12, 4, 1, "fp16", False),        # the guide's 8-rank example
    (4, 2, 8, 64, 1030, 1030, 0, "bf16", False),    # ~21.6 MiB of copies
    (2, 2, 4, 40, 130, 70, 1, "fp16", True),
    (2, 2, 4, 96, 256, 512, 0, "fp16", False),      # TMA-ready: nothing copied
]


def _inputs(case, seed):
    ep, tp, E, C, M, H, t, dt, tr = case
    cfg = FusedConfig("noalloc", ep=ep, tp=tp, E=E, C=C, M=M, H=H, y_shard_type=t, dtype=dt,
                      seed=seed)
    inp = fused_inputs_host(cfg)
    x = [u.cuda() for u in inp["x"]]
    w = [(u.transpose(1, 2).contiguous() if tr else u).cuda() for u in inp["w"]]
    b = [u.cuda() for u in inp["bias"]]
    return cfg, x, w, b


def _outputs(cfg, dtype):
    ys = bra.bmm_rs_a2a_infer_shape(cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H,
                                    cfg.y_shard_type)["y"]
    return [torch.full(ys, float("nan"), dtype=dtype, device="cuda") for _ in range(cfg.P)]


def _existing(cfg, x, w, b, tr):
    """bmm_rs_a2a_ex, packed variant, workspace from torch's allocator."""
    out = _outputs(cfg, x[0].dtype)
    need = bra.bmm_rs_a2a_workspace_size(x, w, b, cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H,
                                         cfg.y_shard_type, out, transpose_weight=tr)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda") if need > 0 else None
    bra.bmm_rs_a2a(x, w, b, cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, cfg.y_shard_type,
                   out=out, transpose_weight=tr, variant="packed", workspace=ws)
    torch.cuda.synchronize()
    return out, need


def _noalloc_c(cfg, x, w, b, tr):
    """bmm_rs_a2a_noalloc called through the C ABI with ctypes."""
    out = _outputs(cfg, x[0].dtype)
    arr = lambda ts: bra._ptr_array([t.data_ptr() for t in ts])
    code = bra.FP16 if x[0].dtype == torch.float16 else bra.BF16
    rc = bra.library().bmm_rs_a2a_noalloc(
        arr(x), arr(w), arr(b), cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H, cfg.y_shard_type,
        code, arr(out), 1 if tr else 0, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, bra.status_str(rc)
    torch.cuda.synchronize()
    assert bra.fault_status() == 0
    return out


def _rel(a, b):
    g = np.concatenate([t.float().cpu().numpy().astype(np.float64).ravel() for t in a])
    r = np.concatenate([t.float().cpu().numpy().astype(np.float64).ravel() for t in b])
    assert np.isfinite(g).all(), "an output element was not written"
    return float(np.max(np.abs(g - r)) / max(np.max(np.abs(r)), 1e-30))


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES)
def test_noalloc_matches_the_workspace_call_twice(case):
    tr, dt = case[8], case[7]
    for seed in (101, 202):                     # two calls in a row, different inputs
        cfg, x, w, b = _inputs(case, seed + sum(case[:6]))
        ref, need = _existing(cfg, x, w, b, tr)
        assert need <= bra.NOALLOC_SCRATCH_BYTES
        got = _noalloc_c(cfg, x, w, b, tr)
        err = _rel(got, ref)
        assert err <= TOL[dt], f"{case} seed {seed}: rel err {err:.3e}"


def test_noalloc_rejects_copies_beyond_the_scratch_array():
    """Checked on the host before any device call (stand-in pointers)."""
    lib = bra.library()
    f = Fake(8, 2, 16, 16, 2050, 1030, 0)       # ~80 MB of copies
    x, w, b, y = f.arrays()
    need = lib.bmm_rs_a2a_workspace_size(x, w, b, *f.args, bra.FP16, y, None)
    assert need > bra.NOALLOC_SCRATCH_BYTES
    assert lib.bmm_rs_a2a_noalloc(x, w, b, *f.args, bra.FP16, y, 0, None) == UNSUPPORTED
    assert lib.bmm_rs_a2a_noalloc(None, w, b, *f.args, bra.FP16, y, 0, None) == NULLPTR
