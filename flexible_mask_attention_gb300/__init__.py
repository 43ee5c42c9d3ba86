"""Flexible-mask flash attention for NVIDIA GB300 (sm_103a).

Thin binding over the C ABI of ``libffa.so`` (declared in ``include/ffa.h``):
the functions below carry the same names and only marshal arguments.  Every
step of the computation runs in the library's CUDA kernels; PyTorch supplies
device memory and the current stream.  There is no CPU path: if the library
is not built, or no sm_103 device is present, the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

__all__ = [
    "FFA_FULL", "FFA_CAUSAL", "FFA_INV_CAUSAL", "FFA_BI_CAUSAL", "FFAError", "Plan",
    "library_path", "load_library", "ffa_plan_create", "ffa_plan_destroy", "ffa_plan_info",
    "ffa_plan_export", "ffa_fwd_workspace_size", "ffa_bwd_workspace_size", "ffa_fwd", "ffa_bwd",
    "ffa_get_last_device_error", "ffa_plan_set_wait_limit", "ffa_kernel_launch_count",
    "ffa_bwd_noalloc", "ffa_plan_set_events", "ffa_fwd_ex", "ffa_bwd_ex", "FFA_SINK_SH",
    "FFA_SINK_SSH", "FFA_MAX_SINK", "EXPORTED_SYMBOLS",
]

FFA_FULL, FFA_CAUSAL, FFA_INV_CAUSAL, FFA_BI_CAUSAL = 0, 1, 2, 3
FFA_SINK_SH, FFA_SINK_SSH = 0, 1  # sink layouts [n_sink, Hq] and [Tq, n_sink, Hq]
FFA_MAX_SINK = 64
_SINK_LAYOUTS = {"sh": FFA_SINK_SH, "ssh": FFA_SINK_SSH}

_HERE = os.path.dirname(os.path.abspath(__file__))
_STATUS = {0: "ok", 1: "invalid argument", 2: "slice range out of bounds or bad mask type",
           3: "slice rectangles overlap", 4: "unsupported configuration",
           5: "workspace too small", 6: "device wait timed out", 7: "CUDA runtime error"}

EXPORTED_SYMBOLS = [
    "ffa_plan_create", "ffa_plan_destroy", "ffa_plan_info", "ffa_plan_export",
    "ffa_fwd_workspace_size", "ffa_bwd_workspace_size", "ffa_fwd", "ffa_bwd",
    "ffa_get_last_device_error", "ffa_plan_set_wait_limit", "ffa_status_string",
    "ffa_kernel_launch_count", "ffa_bwd_noalloc", "ffa_bwd_noalloc_max_workspace",
    "ffa_plan_set_events", "ffa_fwd_ex", "ffa_bwd_ex",
]


class FFAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {_STATUS.get(status, 'unknown')} (status {status})")
        self.status = status


class _PlanInfo(ctypes.Structure):
    _fields_ = [("fwd_steps", ctypes.c_int64), ("fwd_items", ctypes.c_int64),
                ("bwd_steps", ctypes.c_int64), ("bwd_items", ctypes.c_int64),
                ("merges", ctypes.c_int64), ("grid_fwd", ctypes.c_int32),
                ("grid_bwd", ctypes.c_int32), ("area", ctypes.c_int64),
                ("fwd_masks", ctypes.c_int64), ("bwd_masks", ctypes.c_int64),
                ("gathers", ctypes.c_int64), ("bgathers", ctypes.c_int64),
                ("stacked", ctypes.c_int64)]


_lib = None


def library_path() -> str:
    return os.path.join(_HERE, "_build", "libffa.so")


def load_library():
    """Open libffa.so (built by ``__graft_entry__.build()``) and declare its ABI."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I32, I64, U64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
    F = ctypes.c_float
    S = ctypes.c_size_t
    lib.ffa_plan_create.argtypes = [ctypes.POINTER(P), P, P, P, I32, I32, I32, I32, I32, I32, I32,
                                    I32, P]
    lib.ffa_plan_destroy.argtypes = [P]
    lib.ffa_plan_info.argtypes = [P, ctypes.POINTER(_PlanInfo)]
    lib.ffa_plan_export.argtypes = [P, I32, P, I64, ctypes.POINTER(I64)]
    lib.ffa_fwd_workspace_size.argtypes = [P]
    lib.ffa_fwd_workspace_size.restype = S
    lib.ffa_bwd_workspace_size.argtypes = [P]
    lib.ffa_bwd_workspace_size.restype = S
    lib.ffa_fwd.argtypes = [P, P, P, P, F, P, P, P, S, P]
    lib.ffa_bwd.argtypes = [P, P, P, P, P, P, P, F, P, P, P, P, S, P]
    lib.ffa_fwd_ex.argtypes = [P, P, P, P, P, I32, I32, F, F, P, P, P, S, P]
    lib.ffa_bwd_ex.argtypes = [P, P, P, P, P, P, P, P, I32, I32, F, F, P, P, P, P, P, S, P]
    lib.ffa_get_last_device_error.argtypes = [P, ctypes.POINTER(I32), ctypes.POINTER(I32), P]
    lib.ffa_plan_set_wait_limit.argtypes = [P, U64]
    lib.ffa_plan_set_events.argtypes = [P, ctypes.POINTER(P), I32]
    lib.ffa_status_string.argtypes = [I32]
    lib.ffa_status_string.restype = ctypes.c_char_p
    lib.ffa_kernel_launch_count.argtypes = []
    lib.ffa_kernel_launch_count.restype = U64
    lib.ffa_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, F, P, P, P, P]
    lib.ffa_bwd_noalloc_max_workspace.argtypes = []
    lib.ffa_bwd_noalloc_max_workspace.restype = S
    for name in EXPORTED_SYMBOLS:
        if name not in ("ffa_fwd_workspace_size", "ffa_bwd_workspace_size", "ffa_status_string",
                        "ffa_kernel_launch_count", "ffa_bwd_noalloc_max_workspace"):
            getattr(lib, name).restype = I32
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != 0:
        raise FFAError(fn, status)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


class Plan:
    """Owns an ``ffa_plan_t``: the tile work lists for one slice table and shape."""

    def __init__(self, handle, total_q, total_k, hq, hkv, d, device):
        self._h = handle
        self.total_q, self.total_k = total_q, total_k
        self.num_heads_q, self.num_heads_kv, self.head_dim = hq, hkv, d
        self.device = device

    @property
    def handle(self):
        if self._h is None:
            raise RuntimeError("plan already destroyed")
        return self._h

    def destroy(self):
        if self._h is not None:
            load_library().ffa_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def ffa_plan_create(q_ranges, k_ranges, mask_types, total_q: int, total_k: int,
                    num_heads_q: int, num_heads_kv: int, head_dim: int, num_sms: int = 0,
                    split_below: int = 0, stream=None) -> Plan:
    """Build the work lists for a slice table (ranges [S, 2] int32, types [S] int32)."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    qr = torch.as_tensor(q_ranges, dtype=torch.int32).reshape(-1, 2).to(dev).contiguous()
    kr = torch.as_tensor(k_ranges, dtype=torch.int32).reshape(-1, 2).to(dev).contiguous()
    ty = torch.as_tensor(mask_types, dtype=torch.int32).reshape(-1).to(dev).contiguous()
    if not (qr.shape[0] == kr.shape[0] == ty.shape[0]):
        raise ValueError("q_ranges, k_ranges and mask_types disagree on the slice count")
    h = ctypes.c_void_p()
    _check("ffa_plan_create", lib.ffa_plan_create(
        ctypes.byref(h), _ptr(qr), _ptr(kr), _ptr(ty), int(ty.shape[0]), int(total_q),
        int(total_k), int(num_heads_q), int(num_heads_kv), int(head_dim), int(num_sms),
        int(split_below), _stream(stream)))
    return Plan(h, int(total_q), int(total_k), int(num_heads_q), int(num_heads_kv), int(head_dim),
                dev)


def ffa_plan_destroy(plan: Plan):
    plan.destroy()


def ffa_plan_info(plan: Plan) -> dict:
    info = _PlanInfo()
    _check("ffa_plan_info", load_library().ffa_plan_info(plan.handle, ctypes.byref(info)))
    return {f: getattr(info, f) for f, _ in _PlanInfo._fields_}


_EXPORT_WORDS = {0: 4, 1: 8, 2: 1, 3: 4, 4: 8, 5: 1, 6: 8, 7: 1, 8: 1, 9: 144, 10: 80}


def ffa_plan_export(plan: Plan, which: int):
    """Host copy of one work list as an int32 numpy array of shape [n, words]."""
    import numpy as np
    lib = load_library()
    n = ctypes.c_int64()
    lib.ffa_plan_export(plan.handle, int(which), None, 0, ctypes.byref(n))
    buf = np.zeros(max(1, n.value), dtype=np.int32)
    _check("ffa_plan_export", lib.ffa_plan_export(
        plan.handle, int(which), buf.ctypes.data_as(ctypes.c_void_p), int(buf.size),
        ctypes.byref(n)))
    return buf[: n.value].reshape(-1, _EXPORT_WORDS[which])


def ffa_fwd_workspace_size(plan: Plan) -> int:
    return int(load_library().ffa_fwd_workspace_size(plan.handle))


def ffa_bwd_workspace_size(plan: Plan) -> int:
    return int(load_library().ffa_bwd_workspace_size(plan.handle))


def _workspace(nbytes: int, device, workspace):
    if nbytes == 0:
        return None
    if workspace is None:
        return torch.empty(nbytes, dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError("workspace too small")
    return workspace


def ffa_fwd(plan: Plan, q, k, v, out=None, lse=None, softmax_scale=None, workspace=None,
            stream=None):
    """out[Tq, Hq, D] (bf16), lse[Hq, Tq] (fp32) for the plan's mask."""
    Tq, Tk, Hq, Hkv, D = (plan.total_q, plan.total_k, plan.num_heads_q, plan.num_heads_kv,
                          plan.head_dim)
    _need(q, "q", torch.bfloat16, (Tq, Hq, D))
    _need(k, "k", torch.bfloat16, (Tk, Hkv, D))
    _need(v, "v", torch.bfloat16, (Tk, Hkv, D))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(Hq, Tq, dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, (Tq, Hq, D))
    _need(lse, "lse", torch.float32, (Hq, Tq))
    nbytes = ffa_fwd_workspace_size(plan)
    ws = _workspace(nbytes, q.device, workspace)
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check("ffa_fwd", load_library().ffa_fwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), scale,
                                             _ptr(out), _ptr(lse), _ptr(ws), nbytes,
                                             _stream(stream)))
    return out, lse


def ffa_bwd(plan: Plan, q, k, v, out, dout, lse, dq=None, dk=None, dv=None, softmax_scale=None,
            workspace=None, stream=None):
    """dq, dk, dv (bf16) for dL/dout = dout."""
    Tq, Tk, Hq, Hkv, D = (plan.total_q, plan.total_k, plan.num_heads_q, plan.num_heads_kv,
                          plan.head_dim)
    for t, n, s in ((q, "q", (Tq, Hq, D)), (k, "k", (Tk, Hkv, D)), (v, "v", (Tk, Hkv, D)),
                    (out, "out", (Tq, Hq, D)), (dout, "dout", (Tq, Hq, D))):
        _need(t, n, torch.bfloat16, s)
    _need(lse, "lse", torch.float32, (Hq, Tq))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n, s in ((dq, "dq", (Tq, Hq, D)), (dk, "dk", (Tk, Hkv, D)), (dv, "dv", (Tk, Hkv, D))):
        _need(t, n, torch.bfloat16, s)
    nbytes = ffa_bwd_workspace_size(plan)
    ws = _workspace(nbytes, q.device, workspace)
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check("ffa_bwd", load_library().ffa_bwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                             _ptr(dout), _ptr(lse), scale, _ptr(dq), _ptr(dk),
                                             _ptr(dv), _ptr(ws), nbytes, _stream(stream)))
    return dq, dk, dv


def _sink_args(plan: Plan, sink, sink_layout):
    """(pointer, num_sink, layout code) of an optional fp32 sink tensor."""
    if sink is None:
        return None, 0, FFA_SINK_SH
    if sink_layout not in _SINK_LAYOUTS:
        raise ValueError("sink_layout must be 'sh' or 'ssh'")
    code = _SINK_LAYOUTS[sink_layout]
    Tq, Hq = plan.total_q, plan.num_heads_q
    if not (sink.is_cuda and sink.dtype == torch.float32 and sink.is_contiguous()):
        raise ValueError("sink must be a contiguous fp32 CUDA tensor")
    if code == FFA_SINK_SH and (sink.dim() != 2 or sink.shape[1] != Hq):
        raise ValueError(f"sink layout 'sh' wants [n_sink, {Hq}], got {tuple(sink.shape)}")
    if code == FFA_SINK_SSH and (sink.dim() != 3 or sink.shape[0] != Tq or sink.shape[2] != Hq):
        raise ValueError(f"sink layout 'ssh' wants [{Tq}, n_sink, {Hq}], got {tuple(sink.shape)}")
    return _ptr(sink), int(sink.shape[-2]), code


def ffa_fwd_ex(plan: Plan, q, k, v, sink=None, sink_layout="sh", out=None, lse=None,
               softmax_scale=None, softcap=0.0, workspace=None, stream=None):
    """ffa_fwd with optional attention-sink logits (fp32, [n_sink, Hq] for
    "sh" or [Tq, n_sink, Hq] for "ssh"; lse includes the sink term) and an
    optional softcap c > 0 (scores become c * tanh(score / c))."""
    Tq, Tk, Hq, Hkv, D = (plan.total_q, plan.total_k, plan.num_heads_q, plan.num_heads_kv,
                          plan.head_dim)
    _need(q, "q", torch.bfloat16, (Tq, Hq, D))
    _need(k, "k", torch.bfloat16, (Tk, Hkv, D))
    _need(v, "v", torch.bfloat16, (Tk, Hkv, D))
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(Hq, Tq, dtype=torch.float32, device=q.device) if lse is None else lse
    _need(out, "out", torch.bfloat16, (Tq, Hq, D))
    _need(lse, "lse", torch.float32, (Hq, Tq))
    sp, ns, lay = _sink_args(plan, sink, sink_layout)
    nbytes = ffa_fwd_workspace_size(plan)
    ws = _workspace(nbytes, q.device, workspace)
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check("ffa_fwd_ex", load_library().ffa_fwd_ex(plan.handle, _ptr(q), _ptr(k), _ptr(v), sp, ns,
                                                   lay, scale, float(softcap), _ptr(out), _ptr(lse),
                                                   _ptr(ws), nbytes, _stream(stream)))
    return out, lse


def ffa_bwd_ex(plan: Plan, q, k, v, out, dout, lse, sink=None, sink_layout="sh", dq=None,
               dk=None, dv=None, dsink=None, softmax_scale=None, softcap=0.0, workspace=None,
               stream=None):
    """Backward of ffa_fwd_ex: (dq, dk, dv, dsink); dsink is None without a sink."""
    Tq, Tk, Hq, Hkv, D = (plan.total_q, plan.total_k, plan.num_heads_q, plan.num_heads_kv,
                          plan.head_dim)
    for t, n, s in ((q, "q", (Tq, Hq, D)), (k, "k", (Tk, Hkv, D)), (v, "v", (Tk, Hkv, D)),
                    (out, "out", (Tq, Hq, D)), (dout, "dout", (Tq, Hq, D))):
        _need(t, n, torch.bfloat16, s)
    _need(lse, "lse", torch.float32, (Hq, Tq))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n, s in ((dq, "dq", (Tq, Hq, D)), (dk, "dk", (Tk, Hkv, D)), (dv, "dv", (Tk, Hkv, D))):
        _need(t, n, torch.bfloat16, s)
    sp, ns, lay = _sink_args(plan, sink, sink_layout)
    if ns > 0 and dsink is None:
        dsink = torch.empty_like(sink)
    if dsink is not None:
        _need(dsink, "dsink", torch.float32, tuple(sink.shape))
    nbytes = ffa_bwd_workspace_size(plan)
    ws = _workspace(nbytes, q.device, workspace)
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check("ffa_bwd_ex", load_library().ffa_bwd_ex(
        plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), sp, ns, lay,
        scale, float(softcap), _ptr(dq), _ptr(dk), _ptr(dv), None if dsink is None else _ptr(dsink),
        _ptr(ws), nbytes, _stream(stream)))
    return dq, dk, dv, (dsink if ns > 0 else None)


def ffa_bwd_noalloc(plan: Plan, q, k, v, out, dout, lse, dq, dk, dv, softmax_scale=None,
                    stream=None):
    """ffa_bwd with the library's fixed scratch array: passes no workspace and
    makes the library allocate nothing (outputs must be given)."""
    Tq, Tk, Hq, Hkv, D = (plan.total_q, plan.total_k, plan.num_heads_q, plan.num_heads_kv,
                          plan.head_dim)
    for t, n, s in ((q, "q", (Tq, Hq, D)), (k, "k", (Tk, Hkv, D)), (v, "v", (Tk, Hkv, D)),
                    (out, "out", (Tq, Hq, D)), (dout, "dout", (Tq, Hq, D)),
                    (dq, "dq", (Tq, Hq, D)), (dk, "dk", (Tk, Hkv, D)), (dv, "dv", (Tk, Hkv, D))):
        _need(t, n, torch.bfloat16, s)
    _need(lse, "lse", torch.float32, (Hq, Tq))
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check("ffa_bwd_noalloc", load_library().ffa_bwd_noalloc(
        plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), scale,
        _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)))
    return dq, dk, dv


def ffa_get_last_device_error(plan: Plan, stream=None):
    """(code, where) of the first device-side failure since the last call; clears it."""
    code, where = ctypes.c_int32(), ctypes.c_int32()
    _check("ffa_get_last_device_error", load_library().ffa_get_last_device_error(
        plan.handle, ctypes.byref(code), ctypes.byref(where), _stream(stream)))
    return code.value, where.value


def ffa_plan_set_events(plan: Plan, events):
    """Phase events (six torch.cuda.Event with timing) recorded by the library
    around its forward and backward kernels; None stops recording."""
    if events is None:
        _check("ffa_plan_set_events", load_library().ffa_plan_set_events(plan.handle, None, 0))
        plan._events = None
        return
    if len(events) != 6:
        raise ValueError("six events are required")
    for e in events:
        if not e.cuda_event:  # torch creates the event on its first record
            e.record()
    arr = (ctypes.c_void_p * 6)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    plan._events = (events, arr)  # keep the handles alive with the plan
    _check("ffa_plan_set_events", load_library().ffa_plan_set_events(plan.handle, arr, 6))


def ffa_plan_set_wait_limit(plan: Plan, nanoseconds: int):
    _check("ffa_plan_set_wait_limit",
           load_library().ffa_plan_set_wait_limit(plan.handle, int(nanoseconds)))


def ffa_kernel_launch_count() -> int:
    """Kernels the library has launched in this process."""
    return int(load_library().ffa_kernel_launch_count())


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
