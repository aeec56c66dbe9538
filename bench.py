"""Benchmark: fused BMM -> TP ReduceScatter -> Add -> EP AllToAll and all_to_all_v.

One step = one pass of the whole hot path over one batch of synthetic input:
  * bmm_rs_a2a on ep=8, tp=4 (32 virtual ranks), E=64, C=512, M=8192, H=4096,
    yShardType 1, fp16 (17.59 TFLOP, 8.6 GB of inputs), then
  * all_to_all_v on int8, P=32, L=64 (B=64), Dirichlet(0.3)-skewed counts,
    about 2 MiB sent per rank.
Inputs are resident in HBM before the timed region; both are larger than L2
or evicted by the fused call's 10 GB of traffic between all_to_all_v calls.

Prints one JSON line (rank 0).  Besides the step it reports all_to_all_v and
the indexed exchange (each sender's list a permutation of its input) timed
alone, the same op unfused from torch ops as context, and an end-to-end figure
with host buffers.  `--fused NAME` picks another fused workload and
`--workspace` gives the fused call a workspace (unaligned shapes then time the
packed variant).  `--impl reference` times the CPU oracle on a bounded
sample of the same workload instead.  With torchrun (N > 1) every
rank runs an independent replica of the step on its own GPU.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FUSED_NAME = "ep8tp4_E64_C512_M8192_H4096_t1_fp16"
A2AV_NAME = "P32_L64_int8_dirichlet0.3"
METRIC = "fused BMM-RS-A2A TFLOP/s & all_to_all_v GB/s (1 GB300) vs roofline"


def _args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-unfused", action="store_true",
                    help="skip the unfused torch (cuBLAS bmm + elementwise) context timing")
    ap.add_argument("--a2av-alone-calls", type=int, default=30,
                    help="all_to_all_v calls timed alone after the step loop (0: none)")
    ap.add_argument("--indexed-calls", type=int, default=30,
                    help="indexed all_to_all_v calls timed alone after the step loop (0: none)")
    ap.add_argument("--fused", default=FUSED_NAME)
    ap.add_argument("--workspace", action="store_true",
                    help="give the fused call a workspace of bmm_rs_a2a_workspace_size bytes: "
                         "shapes whose x or weight rows lack a 16-byte pitch then run the "
                         "packed variant (operands repacked, then the TMA kernel)")
    ap.add_argument("--a2av", default=A2AV_NAME)
    ap.add_argument("--a2av-scale", type=int, default=None,
                    help="counts scale of the Dirichlet exchange workload (its counts are "
                         "rint(scale * w_ij); the default 2^21 sends ~2 MiB per rank)")
    ap.add_argument("--a2av-sweep", action="store_true",
                    help="instead of the step: all_to_all_v alone over a range of sizes "
                         "(L2 swept before every timed call), plus a CUDA graph of 100 "
                         "back-to-back calls per size; one JSON line per size")
    ap.add_argument("--mma-peak", action="store_true",
                    help="instead of the step: the tensor-core rate probe on every SM (dense "
                         "kind::f16 FLOP per SM clock) and the peak it implies")
    ap.add_argument("--sweep-core-num", type=int, nargs="*", default=None,
                    help="core_num values for --a2av-sweep (default: each workload's L)")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------
# distributed plumbing (barrier + max over ranks; no data-path collective)
# --------------------------------------------------------------------------

class Dist:
    def __init__(self, backend=None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            if not dist.is_initialized():
                dist.init_process_group(backend=backend or "nccl")
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float, device=None) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, v: float, device=None) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def aggregate(dist: Dist, per_rank_units: float, per_rank_seconds: float, device=None):
    """Whole-job throughput: units all ranks processed / the slowest rank's time."""
    total_units = dist.sum(per_rank_units, device)
    t = dist.max(per_rank_seconds, device)
    return total_units / t, t


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []           # (monotonic arrival time, fields)
        self.proc = None
        self.thread = None
        self.window = None       # (t0, t1) of the timed region

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.monotonic(), [x.strip() for x in line.split(",")]))

    def mark(self, t0: float, t1: float):
        self.window = (t0, t1)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = self.rows
        if self.window is not None:
            inside = [r for t, r in rows if self.window[0] <= t <= self.window[1]]
            rows = inside if inside else [r for _, r in rows]
        else:
            rows = [r for _, r in rows]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                power.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for k, name in enumerate(names):
                if len(r) > 5 + k and r[5 + k].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def _a2av_config(a):
    from workloads import A2AV_CONFIGS
    cfg = A2AV_CONFIGS[a.a2av]
    if a.a2av_scale is not None:
        if cfg.counts != "dirichlet":
            raise SystemExit("--a2av-scale applies to a Dirichlet exchange workload")
        cfg = cfg.replace(scale=a.a2av_scale)
    return cfg


def _a2av_name(a):
    """The exchange workload's name, with its counts scale when it was changed."""
    return a.a2av if a.a2av_scale is None else f"{a.a2av}_scale{a.a2av_scale}"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


def _traffic_record(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (same source digest)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        from bmm_reducescatter_alltoall_gb300 import _build
        rec = d.get(kernel)
        if rec and rec.get("source_digest") == _build.source_digest(kernel):
            return rec
    except (OSError, ValueError, KeyError):
        return None
    return None


def _cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# --------------------------------------------------------------------------
# CPU oracle legs (the one place bench.py runs oracle/)
# --------------------------------------------------------------------------

def oracle_fused_sample(cfg, x_host, w_host, b_host):
    """Time the oracle on one local expert per rank (E' = ep) of the workload.
    Returns (flops, seconds)."""
    from oracle import fused as of
    El1 = cfg.replace(E=cfg.ep)
    t0 = time.perf_counter()
    of.bmm_rs_a2a(x_host, w_host, b_host, El1.ep, El1.tp, El1.E, El1.C, El1.M, El1.H,
                  El1.y_shard_type, El1.dtype)
    dt = time.perf_counter() - t0
    return El1.flops, dt


def oracle_a2av(sc, inputs):
    import numpy as np
    from oracle import a2av as oa
    cols = sc.sum(axis=0)
    init = [np.zeros(int(c), dtype=inputs[0].dtype) for c in cols]
    t0 = time.perf_counter()
    oa.all_to_all_v(inputs, sc, init)
    dt = time.perf_counter() - t0
    nbytes = 2 * int(sc.sum()) * inputs[0].itemsize + 4 * sc.size * 8
    return nbytes, dt


def _fused_sample_inputs_host(cfg):
    """Host copies of local expert 0 of every rank, drawn like the full inputs."""
    import torch
    from workloads import fused_inputs_device
    if torch.cuda.is_available():
        dinp = fused_inputs_device(cfg.replace(E=cfg.ep), device="cuda")
        return ([t.cpu() for t in dinp["x"]], [t.cpu() for t in dinp["w"]],
                None if dinp["bias"] is None else [t.cpu() for t in dinp["bias"]])
    from workloads import fused_inputs_host
    h = fused_inputs_host(cfg.replace(E=cfg.ep))
    return h["x"], h["w"], h["bias"]


def run_reference(a):
    """The CPU oracle as it stands, timed on the host cores (rank 0 only).

    Each step is a bounded sample of the workload: one local expert per rank
    (E' = ep) and C' tokens per EP block, C' chosen from a calibration step so
    the whole run takes about 90 s of CPU time; plus the full all_to_all_v.
    """
    dist = Dist(backend="gloo")
    if dist.rank != 0:
        dist.close()
        return
    from workloads import A2AV_CONFIGS, FUSED_CONFIGS, a2av_inputs
    cfg = FUSED_CONFIGS[a.fused]
    acfg = _a2av_config(a)
    sc, inputs = a2av_inputs(acfg)
    # calibrate on a small C', then size C' for the run
    c_small = max(cfg.tp, 64 - 64 % cfg.tp)
    probe = cfg.replace(C=c_small)
    xs, ws, bs = _fused_sample_inputs_host(probe)
    f0, t0 = oracle_fused_sample(probe, xs, ws, bs)
    rate = f0 / max(t0, 1e-6)                       # flop/s of the oracle here
    budget = 90.0 / max(1, a.steps + a.warmup)      # seconds per step
    c_fit = int(budget * rate / f0 * c_small)
    C1 = max(c_small, min(cfg.C, c_fit - c_fit % cfg.tp))
    samp = cfg.replace(C=C1)
    xs, ws, bs = _fused_sample_inputs_host(samp)
    times, flops = [], 0
    for k in range(a.warmup + a.steps):
        f, tf = oracle_fused_sample(samp, xs, ws, bs)
        _, ta = oracle_a2av(sc, inputs)
        if k >= a.warmup:
            times.append(tf + ta)
            flops = f
    step_s = sum(times) / len(times)
    value = flops / step_s / 1e12
    sample = (f"fused oracle (fp64 numpy) on one local expert per rank and C'={C1} tokens per "
              f"EP block ({flops / 1e12:.3f} TFLOP) of {a.fused}, plus the full all_to_all_v "
              f"{_a2av_name(a)}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{a.fused} + {_a2av_name(a)}", "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": _cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    dist.close()


# --------------------------------------------------------------------------
# Context: the same op unfused, from torch ops (cuBLAS bmm per rank, the tp
# sum, the bias add and the all-to-all as copies).  Measurement only; the
# intermediate tensors temp1 / temp2 / temp3 are materialised as the
# reference op's dataflow describes.
# --------------------------------------------------------------------------

def unfused_torch(cfg, x, w, bias, out):
    import torch
    ep, tp, El, C, H, t_ = cfg.ep, cfg.tp, cfg.E // cfg.ep, cfg.C, cfg.H, cfg.y_shard_type
    Hp, Cp = H // tp, C // tp
    for s in range(ep):
        temp2 = None
        for t in range(tp):
            temp1 = torch.bmm(x[s * tp + t], w[s * tp + t])            # (El, ep*C, H)
            temp2 = temp1 if temp2 is None else temp2.add_(temp1)       # the reduce-scatter's sum
        for t in range(tp):
            r = s * tp + t
            if t_ == 0:
                chunk = temp2[:, :, t * Hp:(t + 1) * Hp]                # (El, ep*C, Hp)
                b = None if bias is None else bias[r].reshape(El, 1, Hp)
            else:
                chunk = temp2.view(El, ep, tp, Cp, H)[:, :, t]          # (El, ep, Cp, H)
                b = None if bias is None else bias[r].reshape(El, 1, 1, H)
            temp3 = chunk if b is None else (chunk.float() + b.float()).to(chunk.dtype)
            for j in range(ep):
                blk = temp3[:, j * C:(j + 1) * C] if t_ == 0 else temp3[:, j]
                out[j * tp + t][s * El:(s + 1) * El].copy_(blk)


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def run_ours(a):
    import numpy as np
    import torch

    dist = Dist()
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    from bmm_reducescatter_alltoall_gb300 import _build
    _build.build()
    import bmm_reducescatter_alltoall_gb300 as bra
    from workloads import A2AV_CONFIGS, FUSED_CONFIGS, a2av_index, a2av_inputs, fused_inputs_device

    cfg = FUSED_CONFIGS[a.fused]
    acfg = _a2av_config(a)
    P = cfg.P
    stream = torch.cuda.current_stream(dev)

    # ---- inputs resident in HBM ----
    finp = fused_inputs_device(cfg, device=dev)
    ys = bra.bmm_rs_a2a_infer_shape(cfg.ep, cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H,
                                    cfg.y_shard_type)["y"]
    ydt = finp["x"][0].dtype
    yout = [torch.empty(ys, dtype=ydt, device=dev) for _ in range(P)]
    sc, a_inputs = a2av_inputs(acfg)
    cols = sc.sum(axis=0)
    a_in = [torch.from_numpy(v).to(dev) for v in a_inputs]
    a_out = [torch.empty(int(c), dtype=a_in[0].dtype, device=dev) for c in cols]
    sc_d = torch.from_numpy(sc).to(dev)
    book = [torch.empty((acfg.P, acfg.P), dtype=torch.int64, device=dev) for _ in range(3)]
    # read-only L2 sweep (2x L2) between the two kernels: all_to_all_v starts
    # with its inputs in HBM and no dirty lines of the fused output in L2
    sweep = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    fused_launches = (cfg.ep + max(1, 64 // cfg.tp) - 1) // max(1, 64 // cfg.tp)
    ws_bytes = 0
    workspace = None
    if a.workspace:
        ws_bytes = bra.bmm_rs_a2a_workspace_size(finp["x"], finp["w"], finp["bias"], cfg.ep,
                                                 cfg.tp, cfg.E, cfg.C, cfg.M, cfg.H,
                                                 cfg.y_shard_type, yout)
        if ws_bytes > 0:
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    variant = bra.bmm_rs_a2a_variant(finp["x"], finp["w"], finp["bias"], cfg.ep, cfg.tp, cfg.E,
                                     cfg.C, cfg.M, cfg.H, cfg.y_shard_type, yout,
                                     workspace=workspace)
    names = {bra.VARIANT_TC: "fused_tc_kernel", bra.VARIANT_TC2: "fused_tc2_kernel",
             bra.VARIANT_TCU: "fused_tcu_kernel", bra.VARIANT_TCR: "fused_tcr_kernel",
             bra.VARIANT_SIMT: "fused_simt_kernel"}
    if variant == bra.VARIANT_PACKED:
        # the library's choice between the TMA kernels, restated: the CTA
        # pair with >= 64 pair tiles and > 128 token rows per group
        rows = cfg.ep * cfg.C
        pair_tiles = cfg.E * ((rows + 255) // 256) * ((cfg.H + 255) // 256)
        tma = "fused_tc2_kernel" if pair_tiles >= 64 and rows > 128 else "fused_tc_kernel"
        fused_kernel = "repack_rows_kernel + " + tma
    else:
        fused_kernel = names[variant]

    # prepared calls: the tensors are checked once, each step only calls the library
    fused_plan = bra.bmm_rs_a2a_plan(finp["x"], finp["w"], finp["bias"], cfg.ep, cfg.tp, cfg.E,
                                     cfg.C, cfg.M, cfg.H, cfg.y_shard_type, out=yout,
                                     workspace=workspace)
    a2av_plan = bra.all_to_all_v_plan(a_in, sc_d, a_out, acfg.L, send_displs=book[0],
                                      recv_counts=book[1], recv_displs=book[2])

    def fused():
        fused_plan.run(stream)

    def flush():
        bra.l2_flush(sweep, stream=stream)

    def a2av():
        a2av_plan.run(stream)

    for _ in range(a.warmup):
        fused()
        flush()
        a2av()
    torch.cuda.synchronize(dev)
    if bra.fault_status() != 0:
        raise RuntimeError("watchdog word set during warm-up")

    # ---- timed region ----
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(a.steps)]
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.monotonic()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(a.steps):
        ev[k][0].record(stream)
        fused()
        ev[k][1].record(stream)
        flush()
        ev[k][2].record(stream)
        a2av()
        ev[k][3].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.monotonic()
    dist.barrier()
    time.sleep(0.25)
    sampler.mark(wall0, wall1)
    clocks = sampler.stop()
    if bra.fault_status() != 0:
        raise RuntimeError("watchdog word set during the timed region")

    total_s = t_start.elapsed_time(t_end) / 1e3
    fused_ms = [e[0].elapsed_time(e[1]) for e in ev]
    flush_ms = [e[1].elapsed_time(e[2]) for e in ev]
    a2av_ms = [e[2].elapsed_time(e[3]) for e in ev]
    f_ms = statistics.mean(fused_ms)
    a_ms = statistics.mean(a2av_ms)
    step_flops = cfg.flops
    a_bytes = 2 * int(sc.sum()) * a_in[0].element_size() + 4 * sc.size * 8
    value, t_max = aggregate(dist, step_flops * a.steps / 1e12, total_s, dev)
    ms_per_step = t_max / a.steps * 1e3

    peaks = _peaks()
    # A loop of a second or more runs at the power cap, the condition of the
    # sustained peak; only a short burst is compared with the burst peak.
    timed_alone = total_s < 1.0
    tpeak = peaks["bf16_tflops"] if timed_alone else peaks["bf16_tflops_sustained"]
    f_tflops = step_flops / (f_ms / 1e3) / 1e12
    a_gbs = a_bytes / (a_ms / 1e3) / 1e9
    traffic = _traffic_record(fused_kernel)
    a_traffic = _traffic_record("a2av_kernel")
    roofline = {
        "kernel": fused_kernel, "bound": "tensor", "achieved": f_tflops,
        "peak": tpeak, "unit": "TFLOP/s", "frac": f_tflops / tpeak,
        "frac_of_sustained": f_tflops / peaks["bf16_tflops_sustained"],
        "peak_source": f"{peaks['source']} {'burst' if timed_alone else 'sustained'} bf16 "
                       "(fp16 dense rate equals bf16)",
        "traffic": None if traffic is None else traffic["dram_bytes_per_launch"] * fused_launches,
        "algorithmic_flops_per_launch": step_flops / fused_launches,
        "mean_ms": f_ms, "min_ms": min(fused_ms),
    }
    # ---- context: cuBLAS in the fused op's dtype right after the timed region,
    # for as long (a dense 8192^3 GEMM back to back; under a long loop both run
    # at the power cap, and fp16 settles at a lower clock than bf16) ----
    roofline["cublas_same_dtype"] = cublas_context(torch, dev, ydt, min(max(total_s, 0.3), 4.0),
                                                   f_tflops)
    a2av_line = {
        "kernel": "a2av_kernel", "value": a_gbs, "unit": "GB/s", "bound": "hbm",
        "achieved": a_gbs, "peak": peaks["hbm_gbs"], "frac": a_gbs / peaks["hbm_gbs"],
        "traffic": None if a_traffic is None else a_traffic["dram_bytes_per_launch"],
        "algorithmic_bytes_per_launch": a_bytes, "mean_ms": a_ms, "min_ms": min(a2av_ms),
        "B": bra.cal_all_to_all_v_blocks(acfg.P, acfg.L),
        "blocks": bra.all_to_all_v_launch_blocks(acfg.P, acfg.L),
    }

    # ---- context: the same op unfused from torch ops (after the timed region) ----
    unfused = None
    if not a.no_unfused:
        yref = [torch.empty_like(t) for t in yout]
        unfused_torch(cfg, finp["x"], finp["w"], finp["bias"], yref)      # warm-up
        torch.cuda.synchronize(dev)
        u0 = torch.cuda.Event(enable_timing=True)
        u1 = torch.cuda.Event(enable_timing=True)
        u0.record(stream)
        for _ in range(3):
            unfused_torch(cfg, finp["x"], finp["w"], finp["bias"], yref)
        u1.record(stream)
        torch.cuda.synchronize(dev)
        u_ms = u0.elapsed_time(u1) / 3
        diff = max(float((a_.float() - b_.float()).abs().max()) for a_, b_ in zip(yref, yout))
        scale = max(float(b_.float().abs().max()) for b_ in yout)
        unfused = {
            "ms": u_ms, "tflops": step_flops / (u_ms / 1e3) / 1e12,
            "fused_speedup": u_ms / f_ms,
            "max_rel_diff_vs_fused": diff / scale,
            "what": "torch.bmm per rank (cuBLAS) with temp1/temp2/temp3 materialised, the tp "
                    "sum, bias add and the all-to-all as copies; 3 iterations after the timed "
                    "region (context, not a product path)",
        }
        del yref
        torch.cuda.empty_cache()

    # ---- all_to_all_v timed alone: each call after the L2 sweep, with the GPU
    # idle between calls (not following the fused kernel's power draw) ----
    def time_alone(fn):
        ms = []
        for _ in range(a.a2av_alone_calls):
            torch.cuda._sleep(20_000_000)     # keeps the GPU busy so the host runs ahead
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms.append(e0.elapsed_time(e1))
        return ms

    def alone_record(ms, blocks):
        # the mean, not the median: event times come in ~2 us steps at this size
        m = statistics.mean(ms)
        return {"achieved": a_bytes / (m / 1e3) / 1e9, "unit": "GB/s",
                "frac": a_bytes / (m / 1e3) / 1e9 / peaks["hbm_gbs"], "mean_ms": m,
                "min_ms": min(ms), "calls": len(ms), "blocks": blocks}

    a_alone = time_alone(a2av)
    a2av_line["alone"] = None if not a_alone else {
        **alone_record(a_alone, a2av_line["blocks"]),
        "note": "each call after the read-only L2 sweep, timed alone (CUDA events, ~2 us "
                "resolution); the in-step figure above follows the fused kernel at its "
                "power-capped clock, which also slows L2",
    }
    # The floor of that timing: the same event pair around a launch that does
    # nothing (a one-thread kernel, after the same sweep), and the call's rate
    # net of it.  Context beside `alone`, which stays the figure.
    if a_alone:
        floor = statistics.mean(time_alone(lambda: torch.cuda._sleep(1)))
        net = statistics.mean(a_alone) - floor
        a2av_line["alone"]["net_of_event_floor"] = {
            "floor_ms": floor, "achieved": a_bytes / (net / 1e3) / 1e9, "unit": "GB/s",
            "frac": a_bytes / (net / 1e3) / 1e9 / peaks["hbm_gbs"],
            "note": "floor = the mean event-timed span of an empty launch after the same sweep "
                    "(two events plus one kernel launch); rate = bytes / (alone mean - floor)"}
    # Back to back in a CUDA graph (no sweep between calls, 50 calls per
    # replay): event timing without its ~2 us quantum and launch gaps.
    if a_alone:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            a2av_plan.run(side)
        stream.wait_stream(side)
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(g):
            for _ in range(50):
                a2av_plan.run(torch.cuda.current_stream(dev))
        g.replay()
        torch.cuda.synchronize(dev)
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(4):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        gms = g0.elapsed_time(g1) / 200
        a2av_line["alone_graph"] = {
            "mean_ms": gms, "achieved": a_bytes / (gms / 1e3) / 1e9, "unit": "GB/s",
            "frac": a_bytes / (gms / 1e3) / 1e9 / peaks["hbm_gbs"], "calls": 200,
            "note": "200 calls back to back in a CUDA graph, no L2 sweep between them (the "
                    "payload is larger than L2)"}
        del g
    # The same exchange with core_num = the SM count: as many blocks as the
    # launch-width rule admits on the whole GPU (context for the B above).
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if a_alone:
        full_plan = bra.all_to_all_v_plan(a_in, sc_d, a_out, sms, send_displs=book[0],
                                          recv_counts=book[1], recv_displs=book[2])
        full_plan.run(stream)
        a2av_line["alone_whole_gpu"] = {
            **alone_record(time_alone(lambda: full_plan.run(stream)),
                           bra.all_to_all_v_launch_blocks(acfg.P, sms)),
            "core_num": sms,
        }

    # ---- indexed all_to_all_v timed alone: the same counts and payload, each
    # sender's list gathered through a permutation of its input ----
    indexed = None
    if a.indexed_calls > 0:
        perm = a2av_index(sc, [len(v) for v in a_inputs], "perm", seed=acfg.seed)
        ix = [torch.from_numpy(v).to(dev) for v in perm]

        def ia_time(L):
            plan = bra.indexed_all_to_all_v_plan(a_in, ix, sc_d, a_out, L,
                                                 send_displs=book[0], recv_counts=book[1],
                                                 recv_displs=book[2])
            for _ in range(3):
                plan.run(stream)
            ms = []
            for _ in range(a.indexed_calls):
                torch.cuda._sleep(20_000_000)
                flush()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                plan.run(stream)
                e1.record(stream)
                torch.cuda.synchronize(dev)
                ms.append(e0.elapsed_time(e1))
            return ms

        ia_ms = ia_time(acfg.L)
        n_el = int(sc.sum())
        ia_bytes = 2 * n_el * a_in[0].element_size() + 8 * n_el + 4 * sc.size * 8
        m = statistics.mean(ia_ms)
        # core_num L is the exact block count of this call (one block per
        # SM); the same call on every SM for context
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        w_ms = ia_time(sms)
        wm = statistics.mean(w_ms)
        indexed = {
            "kernel": "ia2av_kernel", "workload": f"{_a2av_name(a)}, index = a permutation of each "
                                                  "sender's input (seeded)",
            "bound": "gathers (one random load per element; gather_bound below), reported also "
                     "in GB/s against HBM",
            "achieved": ia_bytes / (m / 1e3) / 1e9, "unit": "GB/s",
            "frac": ia_bytes / (m / 1e3) / 1e9 / peaks["hbm_gbs"], "peak": peaks["hbm_gbs"],
            "algorithmic_bytes_per_launch": ia_bytes, "mean_ms": m, "min_ms": min(ia_ms),
            "calls": len(ia_ms), "blocks": min(acfg.L, sms),
            "whole_gpu": {"core_num": sms, "blocks": sms, "mean_ms": wm,
                          "achieved": ia_bytes / (wm / 1e3) / 1e9,
                          "frac": ia_bytes / (wm / 1e3) / 1e9 / peaks["hbm_gbs"]},
            "note": "bytes = payload read + write + 8-byte index per element + bookkeeping; "
                    "each call after the read-only L2 sweep, timed alone; the gathers are "
                    "random, one 32-byte sector per element",
        }
        # The gathers, not HBM, bound this call: one load per element, each in
        # its own line.  The gather-rate probe on as many SMs, right after,
        # gives the rate the SMs can issue them at.
        gbuf = torch.randint(0, 256, (64 << 20,), dtype=torch.uint8, device=dev)
        gb = gather_rate(bra, torch, dev, gbuf, min(acfg.L, sms))
        gw = gather_rate(bra, torch, dev, gbuf, sms)
        del gbuf
        indexed["gather_bound"] = {
            "what": "random one-byte loads from a 64 MiB buffer (L2-resident) on the same number "
                    "of SMs, right after (bra_gather_rate_probe): one per gathered element",
            "probe_gathers_per_s": gb["gathers_per_s"], "probe_per_sm_clk": gb["per_sm_clk"],
            "probe_mhz": gb["mhz"], "achieved_gathers_per_s": n_el / (m / 1e3),
            "frac": n_el / (m / 1e3) / gb["gathers_per_s"],
            "whole_gpu": {"probe_gathers_per_s": gw["gathers_per_s"],
                          "probe_per_sm_clk": gw["per_sm_clk"],
                          "achieved_gathers_per_s": n_el / (wm / 1e3),
                          "frac": n_el / (wm / 1e3) / gw["gathers_per_s"]},
        }
        del ix
        if bra.fault_status() != 0:
            raise RuntimeError("watchdog word set by the indexed exchange")

    # ---- the tensor-core rate probe: dense FLOP per SM clock, measured, and
    # the peak it gives at the maximum SM clock (after the timed region) ----
    mma = mma_rate(bra, torch, dev, 1 << 12, torch.float16)
    spec = mma["sms"] * (peaks.get("sm_max_mhz") or 2070.0) * 1e6 * mma["flop_per_sm_clk"] / 1e12
    roofline["spec_peak"] = {
        "tflops": spec, "frac": f_tflops / spec,
        "derivation": f"{mma['sms']} SMs x {peaks.get('sm_max_mhz') or 2070.0:.0f} MHz x "
                      f"{mma['flop_per_sm_clk']:.0f} FLOP per SM clock (tcgen05 kind::f16 "
                      "probe, fp16, all SMs)",
        "probe_mhz": mma["probe_mhz"],
    }

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if a.e2e_steps > 0:
        hx = [t.cpu().pin_memory() for t in finp["x"]]
        hw = [t.cpu().pin_memory() for t in finp["w"]]
        hb = None if finp["bias"] is None else [t.cpu().pin_memory() for t in finp["bias"]]
        ha = [torch.from_numpy(v).pin_memory() for v in a_inputs]
        hsc = torch.from_numpy(sc).pin_memory()
        hy = [torch.empty(ys, dtype=ydt).pin_memory() for _ in range(P)]
        hao = [torch.empty(int(c), dtype=a_in[0].dtype).pin_memory() for c in cols]
        h2d = (sum(t.numel() * t.element_size() for t in hx + hw + ha)
               + (0 if hb is None else sum(t.numel() * t.element_size() for t in hb))
               + hsc.numel() * 8)
        d2h = sum(t.numel() * t.element_size() for t in hy + hao)

        # Two device sets, three streams: the uploads of step k+1 and the
        # read-back of step k-1 run while step k's kernels run.  Every step
        # still uploads all of its inputs and reads back all of its outputs;
        # a set is reused only after its previous kernels and read-back end.
        sets = [dict(x=finp["x"], w=finp["w"], b=finp["bias"], a_in=a_in, sc=sc_d, y=yout,
                     a_out=a_out, book=book)]
        sets.append(dict(
            x=[torch.empty_like(t) for t in finp["x"]], w=[torch.empty_like(t) for t in finp["w"]],
            b=None if finp["bias"] is None else [torch.empty_like(t) for t in finp["bias"]],
            a_in=[torch.empty_like(t) for t in a_in], sc=torch.empty_like(sc_d),
            y=[torch.empty_like(t) for t in yout], a_out=[torch.empty_like(t) for t in a_out],
            book=[torch.empty_like(t) for t in book]))
        up = torch.cuda.Stream(dev)
        down = torch.cuda.Stream(dev)

        def upload(dset):
            for d_, h_ in zip(dset["x"], hx):
                d_.copy_(h_, non_blocking=True)
            for d_, h_ in zip(dset["w"], hw):
                d_.copy_(h_, non_blocking=True)
            if hb is not None:
                for d_, h_ in zip(dset["b"], hb):
                    d_.copy_(h_, non_blocking=True)
            for d_, h_ in zip(dset["a_in"], ha):
                d_.copy_(h_, non_blocking=True)
            dset["sc"].copy_(hsc, non_blocking=True)

        for dset in sets:                          # prepared once per device set
            dset["fplan"] = bra.bmm_rs_a2a_plan(dset["x"], dset["w"], dset["b"], cfg.ep, cfg.tp,
                                                cfg.E, cfg.C, cfg.M, cfg.H, cfg.y_shard_type,
                                                out=dset["y"], workspace=workspace)
            dset["aplan"] = bra.all_to_all_v_plan(dset["a_in"], dset["sc"], dset["a_out"],
                                                  acfg.L, send_displs=dset["book"][0],
                                                  recv_counts=dset["book"][1],
                                                  recv_displs=dset["book"][2])

        def compute(dset):
            dset["fplan"].run(stream)
            bra.l2_flush(sweep, stream=stream)
            dset["aplan"].run(stream)

        def download(dset):
            for h_, d_ in zip(hy, dset["y"]):
                h_.copy_(d_, non_blocking=True)
            for h_, d_ in zip(hao, dset["a_out"]):
                h_.copy_(d_, non_blocking=True)

        def run_steps(n):
            ev = {k: [torch.cuda.Event(), torch.cuda.Event(),
                      torch.cuda.Event(enable_timing=True)] for k in range(n)}
            for k in range(n):
                dset = sets[k % 2]
                up_done, comp_done, down_done = ev[k]
                if k >= 2:
                    up.wait_event(ev[k - 2][1])        # its inputs are no longer read
                with torch.cuda.stream(up):
                    upload(dset)
                up_done.record(up)
                stream.wait_event(up_done)
                if k >= 2:
                    stream.wait_event(ev[k - 2][2])    # its outputs were read back
                compute(dset)
                comp_done.record(stream)
                down.wait_event(comp_done)
                with torch.cuda.stream(down):
                    download(dset)
                down_done.record(down)
            return ev

        run_steps(2)
        torch.cuda.synchronize(dev)
        dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(up)
        stream.wait_event(e0)
        down.wait_event(e0)
        evs = run_steps(a.e2e_steps)
        down.wait_event(evs[a.e2e_steps - 1][2])
        e1.record(down)
        torch.cuda.synchronize(dev)
        dist.barrier()
        if bra.fault_status() != 0:
            raise RuntimeError("watchdog word set during the end-to-end steps")
        e2e_val, _ = aggregate(dist, step_flops * a.e2e_steps / 1e12, e0.elapsed_time(e1) / 1e3,
                               dev)
        e2e_s = e0.elapsed_time(e1) / 1e3
        # device time between consecutive read-back ends: the steady step is
        # bound by the host link; single copies that stall show as outliers
        ends = [e0.elapsed_time(evs[k][2]) for k in range(a.e2e_steps)]
        step_ms = [ends[0]] + [b_ - a_ for a_, b_ in zip(ends, ends[1:])]
        e2e = {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": a.e2e_steps,
               "step_ms": [round(v, 2) for v in step_ms],
               "median_step_ms": float(np.median(step_ms)),
               "pipelined": "uploads of step k+1 and read-back of step k-1 overlap step k "
                            "(two device sets, copy streams)",
               "bound": "host link",
               "link_gbs": (h2d + d2h) * a.e2e_steps / e2e_s / 1e9}
        del sets
        del hx, hw, hb, ha, hy, hao

    # ---- CPU oracle baseline on a bounded sample (rank 0, N = 1 only) ----
    cpu_baseline = None
    if dist.rank == 0 and dist.world == 1 and not a.no_cpu_baseline:
        xs = [t[:1].cpu() for t in finp["x"]]
        ws = [t[:1].cpu() for t in finp["w"]]
        bs = None if finp["bias"] is None else [t[:1].cpu() for t in finp["bias"]]
        del finp
        torch.cuda.empty_cache()
        flops, secs = oracle_fused_sample(cfg, xs, ws, bs)
        cpu_baseline = {
            "value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": _cores(),
            "kind": "oracle",
            "sample": f"fused oracle (fp64 numpy) on local expert 0 of every rank: "
                      f"{flops / 1e12:.2f} TFLOP in {secs:.1f} s",
        }
        nb, sa = oracle_a2av(sc, a_inputs)
        cpu_baseline["all_to_all_v"] = {"value": nb / sa / 1e9, "unit": "GB/s",
                                        "sample": f"full {_a2av_name(a)} exchange in {sa:.3f} s"}

    if dist.rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": dist.world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg.dtype, "data": "synthetic",
            "config": {
                "workload": f"{a.fused} + {_a2av_name(a)}",
                "fused": {"ep": cfg.ep, "tp": cfg.tp, "E": cfg.E, "C": cfg.C, "M": cfg.M,
                          "H": cfg.H, "yShardType": cfg.y_shard_type, "dtype": cfg.dtype,
                          "tflop_per_step": step_flops / 1e12, "variant": fused_kernel,
                          "workspace_bytes": ws_bytes},
                "all_to_all_v": {"P": acfg.P, "L": acfg.L, "dtype": acfg.dtype,
                                 "bytes_moved": a_bytes},
                "parallelism": "replicas" if dist.world > 1 else "single GPU, virtual ranks",
                "l2": "fused inputs larger than L2 (8.6 GB per step); a read-only 256 MiB "
                      "sweep (bra_l2_flush, in the step and its time) runs between the fused "
                      "call and all_to_all_v, so all_to_all_v reads its inputs from HBM with no "
                      "dirty fused output left in L2",
                "l2_sweep_ms": statistics.mean(flush_ms),
            },
            "roofline": roofline,
            "all_to_all_v": a2av_line,
            "indexed_all_to_all_v": indexed,
            "unfused_torch": unfused,
            "cpu_baseline": cpu_baseline,
            "e2e": e2e,
            "clocks": clocks,
            "gpu_launches": a.steps * (fused_launches + 2),
        }
        print(json.dumps(line), flush=True)
    dist.close()

# --------------------------------------------------------------------------
# all_to_all_v size sweep (not the step: a measurement of the exchange alone)
# --------------------------------------------------------------------------

# (base workload, field scaled, values): int8 P=32 Dirichlet rows from 64 KiB
# to 32 MiB sent per rank, fp32 P=8 uniform counts from the workload's 4096
# up to 8M per pair.
SWEEP = [
    ("P32_L64_int8_dirichlet0.3", "scale", [1 << 16, 1 << 18, 1 << 21, 1 << 23, 1 << 25]),
    ("P8_L10_fp32_uniform4096", "count_max", [4096, 1 << 16, 1 << 20, 1 << 23]),
]


def run_a2av_sweep(a):
    import torch

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    from bmm_reducescatter_alltoall_gb300 import _build
    _build.build()
    import bmm_reducescatter_alltoall_gb300 as bra
    from workloads import A2AV_CONFIGS, a2av_counts

    peaks = _peaks()
    sweep = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    timed = max(a.steps, 20)
    cases = [(base, field, v, L) for base, field, values in SWEEP for v in values
             for L in (a.sweep_core_num or [A2AV_CONFIGS[base].L])]
    for base, field, v, L in cases:
        cfg = A2AV_CONFIGS[base].replace(**{field: v, "L": L})
        sc = a2av_counts(cfg)
        dt = torch.int8 if cfg.dtype == "int8" else torch.float32
        g = torch.Generator(device=dev)
        g.manual_seed(cfg.seed)
        ins = []
        for i in range(cfg.P):
            n = int(sc[i].sum())
            if dt == torch.int8:
                ins.append(torch.randint(-128, 128, (n,), generator=g, device=dev,
                                         dtype=torch.int8))
            else:
                ins.append(torch.randn(n, generator=g, device=dev))
        outs = [torch.empty(int(c), dtype=dt, device=dev) for c in sc.sum(axis=0)]
        sc_d = torch.from_numpy(sc).to(dev)
        book = [torch.empty((cfg.P, cfg.P), dtype=torch.int64, device=dev)
                for _ in range(3)]

        def call():
            bra.all_to_all_v(ins, sc_d, outs, cfg.L, send_displs=book[0],
                             recv_counts=book[1], recv_displs=book[2])

        for _ in range(max(a.warmup, 3)):
            bra.l2_flush(sweep, stream=stream)
            call()
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(timed)]
        for e0, e1 in ev:
            torch.cuda._sleep(20_000_000)   # keeps the GPU busy so the host runs ahead
            bra.l2_flush(sweep, stream=stream)
            e0.record(stream)
            call()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        us = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in ev)
        med = statistics.median(us)

        # 100 back-to-back calls in one CUDA graph: launch cost amortised,
        # inputs warm in L2 where they fit
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            call()
        stream.wait_stream(side)
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(graph):
            for _ in range(100):
                call()
        graph.replay()
        torch.cuda.synchronize(dev)
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(3):
            graph.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        graph_us = g0.elapsed_time(g1) * 1e3 / 300
        if bra.fault_status() != 0:
            raise RuntimeError("watchdog word set during the sweep")

        nbytes = 2 * int(sc.sum()) * ins[0].element_size() + 4 * sc.size * 8
        gbs = nbytes / (med * 1e-6) / 1e9
        print(json.dumps({
            "sweep": "all_to_all_v", "workload": base, field: v, "P": cfg.P, "L": cfg.L,
            "blocks": bra.all_to_all_v_launch_blocks(cfg.P, cfg.L),
            "dtype": cfg.dtype, "bytes_moved": nbytes, "calls": timed,
            "median_us": med, "min_us": us[0], "GB/s": gbs,
            "frac_of_hbm": gbs / peaks["hbm_gbs"],
            "graph_us_per_call": graph_us,
            "graph_GB/s": nbytes / (graph_us * 1e-6) / 1e9,
            "l2": "256 MiB read-only sweep before every timed call (not in the time); "
                  "the graph replays run back to back without it",
        }), flush=True)
        del ins, outs, sc_d, book, graph
        torch.cuda.empty_cache()


# --------------------------------------------------------------------------
# tensor-core rate probe (not the step: the per-SM dense f16 / bf16 rate)
# --------------------------------------------------------------------------

MMA_FLOP = 2 * 128 * 256 * 16      # one M=128 N=256 K=16 MMA


def cublas_context(torch, dev, dtype, seconds, fused_tflops):
    """torch.matmul of two 8192 x 8192 matrices in `dtype`, back to back for
    about `seconds`, timed by CUDA events, with the median SM clock sampled
    meanwhile; and the fused kernel's rate over it."""
    n = 8192
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    a = torch.randn(n, n, device=dev, generator=g).to(dtype)
    b = torch.randn(n, n, device=dev, generator=g).to(dtype)
    c = torch.empty(n, n, device=dev, dtype=dtype)
    for _ in range(3):
        torch.matmul(a, b, out=c)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.25)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    calls = 0
    w0 = time.monotonic()
    e0.record()
    while time.monotonic() - w0 < seconds:
        for _ in range(8):
            torch.matmul(a, b, out=c)
        calls += 8
        torch.cuda.synchronize(dev)
    e1.record()
    torch.cuda.synchronize(dev)
    w1 = time.monotonic()
    time.sleep(0.25)
    sampler.mark(w0, w1)
    clk = sampler.stop()
    ms = e0.elapsed_time(e1) / calls
    tf = 2.0 * n ** 3 / (ms / 1e3) / 1e12
    del a, b, c
    return {"tflops": tf, "calls": calls, "seconds": round(w1 - w0, 2), "sm_mhz": clk["sm_mhz"],
            "fused_over_cublas": fused_tflops / tf,
            "what": f"torch.matmul {n}^3 {str(dtype).replace('torch.', '')}, back to back right "
                    "after the timed region for as long as it (context: the same power regime)"}


def gather_rate(bra, torch, dev, buf, ctas, iters=128):
    """The gather-rate probe on `ctas` SMs: random one-byte loads per second
    (CUDA events over the launch) and per SM clock (the CTAs' own cycle
    counts, median), and the clock it ran at."""
    bra.gather_rate_probe(buf, ctas, 8)                     # warm-up
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    rec = bra.gather_rate_probe(buf, ctas, iters)
    e1.record()
    torch.cuda.synchronize(dev)
    r = rec.cpu().numpy()
    per_cta = 1024 * iters * 8
    return {"ctas": int(ctas), "gathers_per_s": ctas * per_cta / (e0.elapsed_time(e1) / 1e3),
            "per_sm_clk": float(statistics.median(per_cta / r[:, 0])),
            "mhz": float(statistics.median(r[:, 0] / r[:, 1] * 1e3)),
            "distinct_sms": int(len(set(r[:, 2].tolist())))}


def mma_rate(bra, torch, dev, iters, dtype, ctas=None):
    """Run the probe on `ctas` SMs (default: all); per-SM FLOP per clock
    (median over CTAs), the clock the probe ran at, and the whole launch's
    TFLOP/s by CUDA events."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ctas = ctas or sms
    bra.mma_rate_probe(ctas, 64, dtype)                    # warm-up
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    rec = bra.mma_rate_probe(ctas, iters, dtype)
    e1.record()
    torch.cuda.synchronize(dev)
    r = rec.cpu().numpy()
    if (r[:, 2] != 0).any():
        raise RuntimeError("tensor-core rate probe: a bounded wait ran out")
    flop = iters * 4 * MMA_FLOP
    per_clk = flop / r[:, 0]
    mhz = r[:, 0] / r[:, 1] * 1e3
    return {"ctas": int(ctas), "sms": int(sms), "distinct_sms": int(len(set(r[:, 3].tolist()))),
            "iters": iters, "flop_per_sm_clk": float(statistics.median(per_clk)),
            "flop_per_sm_clk_min": float(per_clk.min()), "probe_mhz": float(statistics.median(mhz)),
            "tflops_events": ctas * flop / (e0.elapsed_time(e1) / 1e3) / 1e12}


def run_mma_peak(a):
    import torch

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    from bmm_reducescatter_alltoall_gb300 import _build
    _build.build()
    import bmm_reducescatter_alltoall_gb300 as bra

    peaks = _peaks()
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    out = {}
    wall0 = time.monotonic()
    for name, dt in (("bf16", torch.bfloat16), ("fp16", torch.float16)):
        out[name] = {"one_sm": mma_rate(bra, torch, dev, 1 << 14, dt, ctas=1),
                     "all_sms": mma_rate(bra, torch, dev, 1 << 14, dt)}
    wall1 = time.monotonic()
    time.sleep(0.25)
    sampler.mark(wall0, wall1)
    clocks = sampler.stop()
    rate = out["bf16"]["all_sms"]["flop_per_sm_clk"]
    sms = out["bf16"]["all_sms"]["sms"]
    max_mhz = peaks.get("sm_max_mhz") or 2070.0
    print(json.dumps({
        "probe": "tcgen05.mma.cta_group::1.kind::f16 M=128 N=256 K=16, operands resident in "
                 "shared memory, one CTA per SM",
        **out,
        "spec_peak_tflops": sms * max_mhz * 1e6 * rate / 1e12,
        "derivation": f"{sms} SMs x {max_mhz:.0f} MHz (maximum SM clock) x {rate:.0f} dense "
                      "FLOP per SM clock (measured, bf16)",
        "measured_peaks": {"bf16_tflops": peaks["bf16_tflops"],
                           "bf16_tflops_sustained": peaks["bf16_tflops_sustained"]},
        "clocks": clocks,
    }), flush=True)


def main(argv=None):
    a = _args(argv)
    if a.impl == "reference":
        run_reference(a)
    elif a.mma_peak:
        run_mma_peak(a)
    elif a.a2av_sweep:
        run_a2av_sweep(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
