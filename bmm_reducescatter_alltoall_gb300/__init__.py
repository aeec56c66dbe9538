"""GB300-native fused MoE BMM -> TP ReduceScatter -> bias Add -> EP AllToAll,
all_to_all_v and its indexed form over virtual ranks on one GPU.

Thin Python binding over libbmmrsa2a.so (the C ABI in include/bmm_rs_a2a.h):
it checks tensors (device, dtype, contiguity), passes their data pointers and
the current CUDA stream, and raises on a non-zero status.  Every step of the
computation runs in the library's CUDA kernels; there is no other code path.
The library is built in-tree by `bmm_reducescatter_alltoall_gb300._build`;
calling into a missing library raises `RuntimeError`.
"""
from __future__ import annotations

import ctypes
import functools
import os
from typing import List, Optional, Sequence

__all__ = [
    "BraError", "FP16", "BF16", "FP32", "INT8", "VARIANT_TC", "VARIANT_TC2", "VARIANT_SIMT",
    "VARIANT_TCU", "VARIANT_TCR", "VARIANT_PACKED", "wait_selftest", "indexed_all_to_all_v",
    "bmm_rs_a2a_workspace_size", "bmm_rs_a2a_noalloc", "NOALLOC_SCRATCH_BYTES",
    "FusedOptions", "library", "library_path", "bmm_rs_a2a", "bmm_rs_a2a_infer_shape",
    "bmm_rs_a2a_variant", "all_to_all_v", "all_to_all_v_checked", "Plan", "bmm_rs_a2a_plan",
    "all_to_all_v_plan", "indexed_all_to_all_v_plan",
    "cal_all_to_all_v_blocks", "all_to_all_v_launch_blocks", "l2_flush", "mma_rate_probe", "gather_rate_probe", "fault_status", "status_str", "version",
]

FP16, BF16, FP32, INT8 = 0, 1, 2, 3
VARIANT_TC, VARIANT_SIMT, VARIANT_TC2, VARIANT_TCU, VARIANT_TCR, VARIANT_PACKED = 1, 2, 3, 4, 5, 6
OK, ERR_NULLPTR, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = (
    0, 161001, 161002, 161003, 161100, 161101)

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "lib", "libbmmrsa2a.so")
_lib = None


class FusedOptions(ctypes.Structure):
    """bra_fused_options of the C header."""
    _fields_ = [("transpose_weight", ctypes.c_int32), ("variant", ctypes.c_int32),
                ("x_pitch", ctypes.c_int32), ("w_pitch", ctypes.c_int32),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_int64),
                ("status", ctypes.c_void_p)]


class BraError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_str(code) if _lib else code} ({code})")
        self.code = code


def library() -> ctypes.CDLL:
    """The loaded native library (loaded on first use)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise RuntimeError(
            f"native library {library_path} is not built; run "
            "`python -m bmm_reducescatter_alltoall_gb300._build` (needs nvcc)")
    lib = ctypes.CDLL(library_path)
    vp, i64, i32, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
    pp = ctypes.POINTER(ctypes.c_void_p)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.bmm_rs_a2a.argtypes = [pp, pp, pp, i64, i64, i64, i64, i64, i64, i64, c_int, pp, vp]
    lib.bmm_rs_a2a.restype = c_int
    optp = ctypes.POINTER(FusedOptions)
    lib.bmm_rs_a2a_ex.argtypes = [pp, pp, pp, i64, i64, i64, i64, i64, i64, i64, c_int, pp, optp, vp]
    lib.bmm_rs_a2a_ex.restype = c_int
    lib.bmm_rs_a2a_variant.argtypes = [pp, pp, pp, i64, i64, i64, i64, i64, i64, i64, c_int, pp,
                                       optp]
    lib.bmm_rs_a2a_variant.restype = c_int
    lib.bmm_rs_a2a_workspace_size.argtypes = lib.bmm_rs_a2a_variant.argtypes
    lib.bmm_rs_a2a_workspace_size.restype = i64
    lib.bmm_rs_a2a_noalloc.argtypes = [pp, pp, pp, i64, i64, i64, i64, i64, i64, i64, c_int, pp,
                                       c_int, vp]
    lib.bmm_rs_a2a_noalloc.restype = c_int
    lib.bmm_rs_a2a_infer_shape.argtypes = [i64] * 7 + [i64p] * 4
    lib.bmm_rs_a2a_infer_shape.restype = c_int
    lib.cal_all_to_all_v_blocks.argtypes = [i64, i64]
    lib.cal_all_to_all_v_blocks.restype = i64
    lib.all_to_all_v_launch_blocks.argtypes = [i64, i64]
    lib.all_to_all_v_launch_blocks.restype = i64
    lib.all_to_all_v.argtypes = [pp, vp, vp, vp, vp, pp, i64, i64, c_int, vp]
    lib.all_to_all_v.restype = c_int
    lib.all_to_all_v_checked.argtypes = [pp, vp, vp, vp, vp, pp, i64, i64, c_int, i64p, vp, vp]
    lib.all_to_all_v_checked.restype = c_int
    lib.indexed_all_to_all_v.argtypes = [pp, i64p, pp, vp, vp, vp, vp, pp, i64, i64, c_int, vp,
                                         vp]
    lib.indexed_all_to_all_v.restype = c_int
    lib.bra_status_str.argtypes = [c_int]
    lib.bra_status_str.restype = ctypes.c_char_p
    lib.bra_l2_flush.argtypes = [vp, ctypes.c_size_t, vp]
    lib.bra_l2_flush.restype = c_int
    lib.bra_fault_status.argtypes = [ctypes.POINTER(i32), c_int]
    lib.bra_fault_status.restype = c_int
    lib.bra_mma_rate_probe.argtypes = [c_int, c_int, c_int, vp, vp]
    lib.bra_mma_rate_probe.restype = c_int
    lib.bra_gather_rate_probe.argtypes = [vp, i64, c_int, c_int, vp, vp]
    lib.bra_gather_rate_probe.restype = c_int
    lib.bra_wait_selftest.argtypes = [c_int, vp, vp]
    lib.bra_wait_selftest.restype = c_int
    lib.bra_version.argtypes = []
    lib.bra_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_str(code: int) -> str:
    return library().bra_status_str(int(code)).decode()


def version() -> str:
    return library().bra_version().decode()


def _check(code: int, what: str) -> None:
    if code != OK:
        raise BraError(code, what)


def _torch():
    import torch
    return torch


def _ptr_array(ptrs: Sequence[Optional[int]]):
    if not ptrs:
        return (ctypes.c_void_p * 1)()
    return (ctypes.c_void_p * len(ptrs))(*[p if p else None for p in ptrs])


def _stream_handle(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev_tensor(t, what: str, dtype=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{what} must be a CUDA tensor (got {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype} (got {t.dtype})")
    return t


def _checked_ptrs(ts, what: str, dtype, shape=None):
    """Data pointers of the CUDA tensors `ts`, after one pass that checks
    device, dtype, contiguity and (when given) shape of each; only when that
    pass fails is the failing entry looked up for the error message."""
    try:
        ok = all(t.is_cuda and t.dtype is dtype and t.is_contiguous() and
                 (shape is None or t.shape == shape) for t in ts)
    except AttributeError:
        ok = False
    if not ok:
        for r, t in enumerate(ts):
            _dev_tensor(t, f"{what}[{r}]", dtype)
            if shape is not None:
                _shape_check(t, shape, f"{what}[{r}]")
    return [t.data_ptr() for t in ts]


def _pitched_ptrs(ts, what: str, dtype, shape):
    """Data pointers and the shared row pitch (elements; 0 = dense) of 3-D
    CUDA tensors of `shape` that are contiguous or row-pitched: strides
    (shape[1] * pitch, pitch, 1) with pitch >= shape[2], the same pitch for
    every entry (a (d0, d1, pitch) buffer viewed as (d0, d1, d2))."""
    try:
        if all(t.is_cuda and t.dtype is dtype and t.is_contiguous() and t.shape == shape
               for t in ts):
            return [t.data_ptr() for t in ts], 0
    except AttributeError:
        pass
    torch = _torch()
    pitch = None
    for r, t in enumerate(ts):
        name = f"{what}[{r}]"
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
        _shape_check(t, shape, name)
        if t.is_contiguous():
            p = shape[2]
        else:
            # Strides of unit dimensions do not address anything: with d1 = 1
            # the pitch is the step between d0 entries.
            d0, d1, d2 = shape
            s0, s1, s2 = t.stride()
            p = s1 if d1 > 1 else s0
            if not ((d2 == 1 or s2 == 1) and p >= d2 and
                    (d0 == 1 or s0 == d1 * p) and (d1 == 1 or s1 == p)):
                raise ValueError(f"{name} must be contiguous or row-pitched (strides "
                                 f"(d1 * pitch, pitch, 1), pitch >= {shape[2]}); got {t.stride()}")
            if p > 2**31 - 1:
                raise ValueError(f"{name}: row pitch {p} elements exceeds the library's "
                                 f"32-bit pitch field")
        if pitch is None:
            pitch = p
        elif p != pitch:
            raise ValueError(f"every {what} entry must have the same row pitch")
    return [t.data_ptr() for t in ts], (0 if pitch == shape[2] else pitch)


def _fused_dtype(dt) -> int:
    torch = _torch()
    if dt == torch.float16:
        return FP16
    if dt == torch.bfloat16:
        return BF16
    raise TypeError(f"fused op takes float16 or bfloat16, got {dt}")


@functools.lru_cache(maxsize=256)
def _infer_shape(ep, tp, E, C, M, H, y_shard_type) -> tuple:
    arrs = [(ctypes.c_int64 * 3)() for _ in range(4)]
    _check(library().bmm_rs_a2a_infer_shape(ep, tp, E, C, M, H, y_shard_type, *arrs),
           "bmm_rs_a2a_infer_shape")
    return tuple(tuple(a) for a in arrs)


def bmm_rs_a2a_infer_shape(ep, tp, E, C, M, H, y_shard_type) -> dict:
    """Per-rank shapes: {'x','w','bias','y'} as tuples (bias in 3-D form)."""
    return dict(zip(("x", "w", "bias", "y"),
                    _infer_shape(int(ep), int(tp), int(E), int(C), int(M), int(H),
                                 int(y_shard_type))))


def _shape_check(t, want, what):
    if tuple(t.shape) != tuple(want):
        raise ValueError(f"{what} has shape {tuple(t.shape)}, expected {tuple(want)}")


_VARIANTS = {None: 0, "auto": 0, "tc": VARIANT_TC, "tc2": VARIANT_TC2, "simt": VARIANT_SIMT,
             "tcu": VARIANT_TCU, "tcr": VARIANT_TCR, "packed": VARIANT_PACKED}


def _options(transpose_weight: bool, variant, workspace=None, pitches=(0, 0),
             status=None) -> "FusedOptions":
    if variant not in _VARIANTS:
        raise ValueError(f"variant must be one of {sorted(k for k in _VARIANTS if k)}")
    o = FusedOptions()
    o.transpose_weight = 1 if transpose_weight else 0
    o.variant = _VARIANTS[variant]
    o.x_pitch, o.w_pitch = pitches
    if isinstance(workspace, str):
        raise ValueError('workspace="auto" is taken by bmm_rs_a2a and bmm_rs_a2a_plan only')
    if workspace is not None:
        if not (workspace.is_cuda and workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor")
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    if status is not None:
        torch = _torch()
        if not (isinstance(status, torch.Tensor) and status.is_cuda and
                status.dtype == torch.int32 and status.numel() >= 1):
            raise ValueError("status must be a CUDA int32 tensor of at least one element")
        o.status = status.data_ptr()
    return o


def _fused_args(x, weight, bias, ep, tp, E, C, M, H, y_shard_type, out,
                transpose_weight=False):
    P = ep * tp
    if len(x) != P or len(weight) != P:
        raise ValueError(f"x and weight need ep*tp = {P} entries")
    shapes = bmm_rs_a2a_infer_shape(ep, tp, E, C, M, H, y_shard_type)
    wshape = shapes["w"]
    if transpose_weight:                      # stored as (El, H, Kp)
        wshape = (wshape[0], wshape[2], wshape[1])
    dt = x[0].dtype
    xs, xpitch = _pitched_ptrs(x, "x", dt, shapes["x"])
    ws, wpitch = _pitched_ptrs(weight, "weight", dt, tuple(wshape))
    bptr = None
    if bias is not None:
        if len(bias) != P:
            raise ValueError(f"bias needs ep*tp = {P} entries")
        torch = _torch()
        bdt = torch.float16 if dt == torch.float16 else torch.float32
        b3 = shapes["bias"]
        b2 = (b3[0], b3[2])
        ptrs = []
        for r, b in enumerate(bias):
            if b is None:
                ptrs.append(0)
                continue
            if not (b.is_cuda and b.dtype is bdt and b.is_contiguous() and
                    (b.shape == b3 or b.shape == b2)):
                _dev_tensor(b, f"bias[{r}]", bdt)
                raise ValueError(f"bias[{r}] has shape {tuple(b.shape)}, expected {b3} "
                                 f"or {b2}")
            ptrs.append(b.data_ptr())
        bptr = _ptr_array(ptrs)
    if len(out) != P:
        raise ValueError(f"out needs ep*tp = {P} entries")
    ys = _checked_ptrs(out, "out", dt, shapes["y"])
    return (_ptr_array(xs), _ptr_array(ws), bptr, _ptr_array(ys), _fused_dtype(dt),
            (xpitch, wpitch))


class Plan:
    """A library call prepared once.

    The tensors were checked and their data pointers taken when the plan was
    made; run() (or calling the plan) only calls the library, so repeated
    calls on the same buffers skip the per-tensor checks of the one-shot
    functions.  The plan keeps its tensors alive; they must keep their
    storage between runs (no resize or reallocation), while their values may
    change.  run() returns `result` (the outputs) and is asynchronous on
    `stream` (default: the current stream).
    """

    def __init__(self, fn, args, name: str, result, keep):
        self._fn, self._args, self._name = fn, args, name
        self.result = result
        self._keep = keep

    def run(self, stream=None):
        _check(self._fn(*self._args, _stream_handle(stream)), self._name)
        return self.result

    __call__ = run


def bmm_rs_a2a_plan(x: Sequence, weight: Sequence, bias: Optional[Sequence], ep: int, tp: int,
                    E: int, C: int, M: int, H: int, y_shard_type: int,
                    out: Optional[Sequence] = None, transpose_weight: bool = False,
                    variant: Optional[str] = None, workspace=None, status=None) -> Plan:
    """bmm_rs_a2a prepared once (see Plan); plan.run() returns out."""
    torch = _torch()
    if out is None:
        ys = bmm_rs_a2a_infer_shape(ep, tp, E, C, M, H, y_shard_type)["y"]
        out = [torch.empty(ys, dtype=x[0].dtype, device=x[0].device) for _ in range(ep * tp)]
    xp, wp, bp, yp, dt, pitches = _fused_args(x, weight, bias, ep, tp, E, C, M, H, y_shard_type,
                                              out, transpose_weight)
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError('workspace must be a CUDA tensor, None or "auto"')
        # torch's caching allocator provides the scratch memory the library
        # asks for (the library itself allocates nothing); none when the
        # operands are already TMA-ready
        n = library().bmm_rs_a2a_workspace_size(
            xp, wp, bp, ep, tp, E, C, M, H, y_shard_type, dt, yp,
            ctypes.byref(_options(transpose_weight, None, None, pitches)))
        if n < 0:
            raise BraError(-n, "bmm_rs_a2a_workspace_size")
        workspace = (torch.empty(n, dtype=torch.uint8, device=x[0].device) if n > 0 else None)
    opts = _options(transpose_weight, variant, workspace, pitches, status)
    args = (xp, wp, bp, ep, tp, E, C, M, H, y_shard_type, dt, yp, ctypes.byref(opts))
    return Plan(library().bmm_rs_a2a_ex, args, "bmm_rs_a2a", out,
                (x, weight, bias, opts, xp, wp, bp, yp, status, workspace))


def bmm_rs_a2a(x: Sequence, weight: Sequence, bias: Optional[Sequence], ep: int, tp: int,
               E: int, C: int, M: int, H: int, y_shard_type: int,
               out: Optional[Sequence] = None, stream=None, transpose_weight: bool = False,
               variant: Optional[str] = None, workspace=None, status=None) -> List:
    """Fused BMM -> ReduceScatter -> Add -> AllToAll over P = ep*tp ranks.

    x[r], weight[r], bias[r] (or bias None) and out[r] are CUDA tensors of
    the shapes `bmm_rs_a2a_infer_shape` gives; out is allocated when None.
    x and weight may also be row-pitched views of wider buffers (strides
    (d1 * pitch, pitch, 1), one pitch per list): with a pitch that is a
    multiple of 8 elements they run on the TMA kernels with no copy.
    transpose_weight: weight[r] is stored as (El, H, Kp) instead of
    (El, Kp, H).  variant: None/"auto", "tc", "tc2", "tcr", "tcu", "simt" or
    "packed".  workspace: an optional contiguous CUDA tensor of at least
    bmm_rs_a2a_workspace_size(...) bytes, or "auto" to have one of that size
    taken from torch's allocator; given one, shapes whose x or weight rows
    lack a 16-byte pitch run the packed variant (operands repacked into it,
    then the TMA kernel).  status: an optional CUDA int32 tensor, this
    call's own timeout word (0 before the kernels; ERR_TIMEOUT if a bounded
    wait of this call gave up), unlike fault_status(), which every call on
    the device shares.  Returns out.  Asynchronous on `stream` (default:
    current stream).  For repeated calls on the same buffers,
    bmm_rs_a2a_plan skips the checks.
    """
    return bmm_rs_a2a_plan(x, weight, bias, ep, tp, E, C, M, H, y_shard_type, out,
                           transpose_weight, variant, workspace, status).run(stream)


# Size of the library's own scratch array used by bmm_rs_a2a_noalloc
# (BRA_NOALLOC_SCRATCH_BYTES of the C header).
NOALLOC_SCRATCH_BYTES = 32 << 20


def bmm_rs_a2a_noalloc(x: Sequence, weight: Sequence, bias: Optional[Sequence], ep: int,
                       tp: int, E: int, C: int, M: int, H: int, y_shard_type: int,
                       out: Sequence, stream=None, transpose_weight: bool = False) -> List:
    """The packed variant with the library's own scratch array instead of a
    workspace (bmm_rs_a2a_noalloc of the C header): for callers that cannot
    allocate device memory.  Allocates nothing, so `out` is required.  The
    copies must fit NOALLOC_SCRATCH_BYTES; calls that overlap on the GPU
    share the array and race.  Returns out."""
    xp, wp, bp, yp, dt, pitches = _fused_args(x, weight, bias, ep, tp, E, C, M, H, y_shard_type,
                                              out, transpose_weight)
    if pitches != (0, 0):
        raise ValueError("bmm_rs_a2a_noalloc takes dense x and weight")
    _check(library().bmm_rs_a2a_noalloc(xp, wp, bp, ep, tp, E, C, M, H, y_shard_type, dt, yp,
                                        1 if transpose_weight else 0, _stream_handle(stream)),
           "bmm_rs_a2a_noalloc")
    return out


def bmm_rs_a2a_workspace_size(x, weight, bias, ep, tp, E, C, M, H, y_shard_type, out=None,
                              transpose_weight: bool = False) -> int:
    """Bytes of workspace the packed variant needs for these tensors (0: none).

    The size depends on x and weight (their shapes and whether each pointer
    is 16-byte aligned); `out` only enters the check that the packed variant
    can take the call (element-aligned outputs).  Without `out`, freshly
    allocated outputs stand in for it.
    """
    if out is None:
        torch = _torch()
        ys = bmm_rs_a2a_infer_shape(ep, tp, E, C, M, H, y_shard_type)["y"]
        out = [torch.empty(ys, dtype=x[0].dtype, device=x[0].device) for _ in range(ep * tp)]
    xp, wp, bp, yp, dt, pitches = _fused_args(x, weight, bias, ep, tp, E, C, M, H, y_shard_type,
                                              out, transpose_weight)
    opts = _options(transpose_weight, None, None, pitches)
    n = library().bmm_rs_a2a_workspace_size(xp, wp, bp, ep, tp, E, C, M, H, y_shard_type, dt,
                                            yp, ctypes.byref(opts))
    if n < 0:
        raise BraError(-n, "bmm_rs_a2a_workspace_size")
    return n


def bmm_rs_a2a_variant(x, weight, bias, ep, tp, E, C, M, H, y_shard_type, out,
                       transpose_weight: bool = False, variant: Optional[str] = None,
                       workspace=None) -> int:
    """The VARIANT_* constant bmm_rs_a2a would run; raises BraError if rejected."""
    xp, wp, bp, yp, dt, pitches = _fused_args(x, weight, bias, ep, tp, E, C, M, H, y_shard_type,
                                              out, transpose_weight)
    opts = _options(transpose_weight, variant, workspace, pitches)
    v = library().bmm_rs_a2a_variant(xp, wp, bp, ep, tp, E, C, M, H, y_shard_type, dt, yp,
                                     ctypes.byref(opts))
    if v < 0:
        raise BraError(-v, "bmm_rs_a2a_variant")
    return v


def cal_all_to_all_v_blocks(P: int, L: int) -> int:
    return int(library().cal_all_to_all_v_blocks(int(P), int(L)))


def all_to_all_v_launch_blocks(P: int, L: int) -> int:
    """Thread blocks (one per SM) all_to_all_v launches on the current device
    for P ranks and core_num L: CalAllToAllVBlocks(P, L), at most the SM
    count."""
    n = int(library().all_to_all_v_launch_blocks(int(P), int(L)))
    if n < 0:
        _check(-n, "all_to_all_v_launch_blocks")
    return n


def _a2av_args(inputs, send_counts, out, send_displs, recv_counts, recv_displs):
    torch = _torch()
    P = len(inputs)
    if len(out) != P:
        raise ValueError("inputs and out need the same number of ranks")
    dt = inputs[0].dtype
    if dt == torch.float32:
        code = FP32
    elif dt == torch.int8:
        code = INT8
    else:
        raise TypeError(f"all_to_all_v takes float32 or int8, got {dt}")
    _checked_ptrs(inputs, "inputs", dt)
    _checked_ptrs(out, "out", dt)
    _dev_tensor(send_counts, "send_counts", torch.int64)
    if tuple(send_counts.shape) != (P, P):
        raise ValueError(f"send_counts must be ({P}, {P})")
    dev = send_counts.device
    mk = lambda t, n: t if t is not None else torch.empty((P, P), dtype=torch.int64, device=dev)
    sd, rc, rd = mk(send_displs, "sd"), mk(recv_counts, "rc"), mk(recv_displs, "rd")
    for t, n in ((sd, "send_displs"), (rc, "recv_counts"), (rd, "recv_displs")):
        _dev_tensor(t, n, torch.int64)
        if tuple(t.shape) != (P, P):
            raise ValueError(f"{n} must be ({P}, {P})")
    return P, code, sd, rc, rd


def all_to_all_v_plan(inputs: Sequence, send_counts, out: Sequence, core_num: int,
                      send_displs=None, recv_counts=None, recv_displs=None) -> Plan:
    """all_to_all_v prepared once (see Plan); plan.run() returns the result dict."""
    P, code, sd, rc, rd = _a2av_args(inputs, send_counts, out, send_displs, recv_counts,
                                     recv_displs)
    ip = _ptr_array([t.data_ptr() for t in inputs])
    op = _ptr_array([t.data_ptr() for t in out])
    args = (ip, send_counts.data_ptr(), sd.data_ptr(), rc.data_ptr(), rd.data_ptr(), op, P,
            int(core_num), code)
    result = {"out": out, "send_displs": sd, "recv_counts": rc, "recv_displs": rd}
    return Plan(library().all_to_all_v, args, "all_to_all_v", result,
                (inputs, send_counts, ip, op))


def all_to_all_v(inputs: Sequence, send_counts, out: Sequence, core_num: int,
                 send_displs=None, recv_counts=None, recv_displs=None, stream=None) -> dict:
    """Variable-count exchange among P = len(inputs) ranks (see the C header).

    send_counts: CUDA int64 (P, P).  out[j] must hold what rank j receives.
    Returns {'out', 'send_displs', 'recv_counts', 'recv_displs'}.
    """
    return all_to_all_v_plan(inputs, send_counts, out, core_num, send_displs, recv_counts,
                             recv_displs).run(stream)


def all_to_all_v_checked(inputs: Sequence, send_counts, out: Sequence, core_num: int,
                         out_capacity: Optional[Sequence[int]] = None, status=None,
                         send_displs=None, recv_counts=None, recv_displs=None,
                         stream=None) -> dict:
    """all_to_all_v plus device-side checks; the int32 status tensor receives
    0 or ERR_INVALID (negative count or over capacity).  out_capacity defaults
    to each out[j]'s length."""
    torch = _torch()
    P, code, sd, rc, rd = _a2av_args(inputs, send_counts, out, send_displs, recv_counts,
                                     recv_displs)
    if out_capacity is None:
        out_capacity = [t.numel() for t in out]
    cap = (ctypes.c_int64 * P)(*[int(c) for c in out_capacity])
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=send_counts.device)
    _dev_tensor(status, "status", torch.int32)
    _check(library().all_to_all_v_checked(
        _ptr_array([t.data_ptr() for t in inputs]), send_counts.data_ptr(), sd.data_ptr(),
        rc.data_ptr(), rd.data_ptr(), _ptr_array([t.data_ptr() for t in out]), P,
        int(core_num), code, cap, status.data_ptr(), _stream_handle(stream)),
        "all_to_all_v_checked")
    return {"out": out, "send_displs": sd, "recv_counts": rc, "recv_displs": rd,
            "status": status}


def indexed_all_to_all_v(inputs: Sequence, index: Sequence, send_counts, out: Sequence,
                         core_num: int, status=None, send_displs=None, recv_counts=None,
                         recv_displs=None, stream=None) -> dict:
    """Indexed exchange (see the C header): rank i sends inputs[i][index[i][k]]
    in the order of its send list, split by send_counts as in all_to_all_v.

    index[i]: CUDA int64 with at least sum_j send_counts[i][j] entries.
    status: optional CUDA int32 (1 element) set to 0, or ERR_INVALID when an
    index was out of range or the call was rejected on the device.
    Returns {'out', 'send_displs', 'recv_counts', 'recv_displs', 'status'}.
    """
    return indexed_all_to_all_v_plan(inputs, index, send_counts, out, core_num, status,
                                     send_displs, recv_counts, recv_displs).run(stream)


def indexed_all_to_all_v_plan(inputs: Sequence, index: Sequence, send_counts, out: Sequence,
                              core_num: int, status=None, send_displs=None, recv_counts=None,
                              recv_displs=None) -> Plan:
    """indexed_all_to_all_v prepared once (see Plan); plan.run() returns the
    result dict."""
    torch = _torch()
    P, code, sd, rc, rd = _a2av_args(inputs, send_counts, out, send_displs, recv_counts,
                                     recv_displs)
    if len(index) != P:
        raise ValueError(f"index has {len(index)} entries for {P} ranks")
    iptrs = _checked_ptrs(index, "index", torch.int64)
    lens = (ctypes.c_int64 * P)(*[t.numel() for t in inputs])
    if status is not None:
        _dev_tensor(status, "status", torch.int32)
    ip = _ptr_array([t.data_ptr() for t in inputs])
    xp = _ptr_array(iptrs)
    op = _ptr_array([t.data_ptr() for t in out])
    args = (ip, lens, xp, send_counts.data_ptr(), sd.data_ptr(), rc.data_ptr(), rd.data_ptr(),
            op, P, int(core_num), code, None if status is None else status.data_ptr())
    result = {"out": out, "send_displs": sd, "recv_counts": rc, "recv_displs": rd,
              "status": status}
    return Plan(library().indexed_all_to_all_v, args, "indexed_all_to_all_v", result,
                (inputs, index, send_counts, status, ip, xp, op, lens))


def l2_flush(buf, stream=None) -> None:
    """Read all of `buf` (a CUDA tensor larger than L2, contents unchanged) so
    that earlier data is evicted from L2."""
    _dev_tensor(buf, "buf")
    _check(library().bra_l2_flush(buf.data_ptr(), buf.numel() * buf.element_size(),
                                  _stream_handle(stream)), "bra_l2_flush")


WAIT_A2AV, WAIT_TC, WAIT_TC_CLUSTER = 0, 1, 2


def wait_selftest(which: str, status, stream=None) -> None:
    """Run one bounded wait that nothing completes with the wait helper of the
    all_to_all_v kernel (which='a2av', ~2 s), of the tensor-core fused
    kernels (which='tc', ~4 s) or the cluster-scope one of the row-class
    kernel (which='tc_cluster', ~4 s).  `status` (CUDA int32, 1 element) receives
    ERR_TIMEOUT and the watchdog word read by fault_status() is set."""
    torch = _torch()
    code = {"a2av": WAIT_A2AV, "tc": WAIT_TC, "tc_cluster": WAIT_TC_CLUSTER}[which]
    _dev_tensor(status, "status", torch.int32)
    _check(library().bra_wait_selftest(code, status.data_ptr(), _stream_handle(stream)),
           "bra_wait_selftest")


def mma_rate_probe(ctas: int, iters: int, dtype=None, stream=None):
    """Tensor-core rate probe (bra_mma_rate_probe of the C header): `ctas`
    CTAs, one per SM, each issuing iters x 4 back-to-back M=128 N=256 K=16
    kind::f16 MMAs.  Returns a CUDA int64 tensor (ctas, 4): cycles, ns,
    status, SM id per CTA (asynchronous on `stream`)."""
    torch = _torch()
    dt = BF16 if dtype is None or dtype == torch.bfloat16 else FP16
    rec = torch.zeros((int(ctas), 4), dtype=torch.int64, device="cuda")
    _check(library().bra_mma_rate_probe(int(ctas), int(iters), dt, rec.data_ptr(),
                                        _stream_handle(stream)), "bra_mma_rate_probe")
    return rec


def gather_rate_probe(buf, ctas: int, iters: int, stream=None):
    """Gather-rate probe (bra_gather_rate_probe of the C header): `ctas` CTAs,
    one per SM, each 1024 threads x iters x 8 random one-byte loads from
    `buf` (a contiguous CUDA tensor whose size in bytes is a power of two).
    Returns a CUDA int64 tensor (ctas, 4): cycles, ns, SM id, byte sum per
    CTA (asynchronous on `stream`)."""
    torch = _torch()
    if not (buf.is_cuda and buf.is_contiguous()):
        raise ValueError("buf must be a contiguous CUDA tensor")
    rec = torch.zeros((int(ctas), 4), dtype=torch.int64, device=buf.device)
    _check(library().bra_gather_rate_probe(buf.data_ptr(), buf.numel() * buf.element_size(),
                                           int(ctas), int(iters), rec.data_ptr(),
                                           _stream_handle(stream)), "bra_gather_rate_probe")
    return rec


def fault_status(clear: bool = False) -> int:
    """The watchdog word (0, or ERR_TIMEOUT if a bounded wait gave up)."""
    v = ctypes.c_int32(0)
    _check(library().bra_fault_status(ctypes.byref(v), 1 if clear else 0), "bra_fault_status")
    return int(v.value)
