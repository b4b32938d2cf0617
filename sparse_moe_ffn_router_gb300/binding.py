"""ctypes binding of the C ABI in include/moe.h (argument marshalling only).

Each function has the name of the C entry point it calls and takes torch CUDA tensors; it
passes their device pointers and the current CUDA stream, and raises MoEError when the
library returns a status other than MOE_OK. Nothing here computes any part of the layer.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass, fields

import torch

from . import build as _build

MOE_STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE", 3: "MOE_ERR_MISALIGNED",
              4: "MOE_ERR_WORKSPACE_TOO_SMALL", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_DEVICE"}
EXPORTED = ["moe_workspace_size", "moe_workspace_init", "moe_route", "moe_forward", "moe_rmsnorm",
            "moe_last_device_error", "moe_workspace_tap", "moe_set_trace", "moe_launch_count", "moe_route_noalloc", "moe_status_string",
            "moe_router_stats", "moe_expert_shadow_size", "moe_forward_host_experts", "moe_forward_host_io",
            "moe_test_set_wait"]
KERNELS = {"router_scores": 0, "router_topk": 1, "dispatch_local": 2, "dispatch_scan": 3, "dispatch_scatter": 4,
           "gate_up": 5, "down": 6, "combine": 7, "rmsnorm": 8, "shared_gate": 9, "gather": 10, "gemm_plan": 11,
           "decode_fused": 12, "router_stats": 13, "fetch_experts": 14,
           "copy_rows": 15}


# moe_dims.flags: router and shared-gate scores rounded to bf16 before ranking and sigmoid
FLAG_BF16_SCORES = 1
# moe_test_set_wait: the signal held back so that a bounded device wait runs out
TEST_SUPPRESS_SCORE = 1
TEST_SUPPRESS_STAGE = 2


class Dims(ctypes.Structure):
    """moe_dims; a dims tuple is (T, H, E, K, I, Is) or (T, H, E, K, I, Is, flags)."""
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("K", ctypes.c_int32), ("I", ctypes.c_int32), ("Is", ctypes.c_int32), ("flags", ctypes.c_int32)]


class CWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("router_w", "router_b", "gate_up", "down", "shared_gate_up",
                                                "shared_down", "shared_gate")]


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_status_string(status)}")


@dataclass
class Weights:
    """One layer's weights (bf16 CUDA tensors, [Out, In] row-major); router_b may be None."""
    router_w: torch.Tensor
    router_b: torch.Tensor | None
    gate_up: torch.Tensor
    down: torch.Tensor
    shared_gate_up: torch.Tensor
    shared_down: torch.Tensor
    shared_gate: torch.Tensor

    @classmethod
    def from_dict(cls, d: dict) -> "Weights":
        return cls(**{f.name: d.get(f.name) for f in fields(cls)})

    def to_c(self) -> CWeights:
        return CWeights(*[_ptr(getattr(self, f.name)) for f in fields(self)])


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True):
    """Load libmoe_gb300.so (building it first when it is absent or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_missing:
                _build.build()
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"CUDA library {_build.LIB} is missing; run build() first")
            lib = ctypes.CDLL(_build.LIB)
            P, S = ctypes.c_void_p, ctypes.c_size_t
            D, W = ctypes.POINTER(Dims), ctypes.POINTER(CWeights)
            st = ctypes.c_int
            lib.moe_workspace_size.restype = S
            lib.moe_workspace_size.argtypes = [D]
            lib.moe_workspace_init.restype = st
            lib.moe_workspace_init.argtypes = [P, S, P]
            lib.moe_route.restype = st
            lib.moe_route.argtypes = [D, P, W, P, P, P, P, P, P, S, P]
            lib.moe_forward.restype = st
            lib.moe_forward.argtypes = [D, P, W, P, P, P, S, P]
            lib.moe_rmsnorm.restype = st
            lib.moe_rmsnorm.argtypes = [D, P, P, ctypes.c_float, P, P]
            lib.moe_last_device_error.restype = st
            lib.moe_last_device_error.argtypes = [P, P]
            lib.moe_workspace_tap.restype = st
            lib.moe_workspace_tap.argtypes = [D, ctypes.c_int, ctypes.POINTER(S), ctypes.POINTER(S)]
            lib.moe_set_trace.restype = st
            lib.moe_set_trace.argtypes = [ctypes.c_int, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.c_int]
            lib.moe_launch_count.restype = ctypes.c_uint64
            lib.moe_launch_count.argtypes = []
            lib.moe_route_noalloc.restype = st
            lib.moe_route_noalloc.argtypes = [D, P, W, P, P, P, P, P, P]
            lib.moe_router_stats.restype = st
            lib.moe_router_stats.argtypes = [D, P, W, P, P, P, P, S, P]
            lib.moe_expert_shadow_size.restype = S
            lib.moe_expert_shadow_size.argtypes = [D]
            lib.moe_forward_host_experts.restype = st
            lib.moe_forward_host_experts.argtypes = [D, P, W, P, P, P, S, P, S, P]
            lib.moe_forward_host_io.restype = st
            lib.moe_forward_host_io.argtypes = [D, P, W, P, P, P, P, P, S, P]
            lib.moe_test_set_wait.restype = st
            lib.moe_test_set_wait.argtypes = [ctypes.c_uint64, ctypes.c_int]
            lib.moe_status_string.restype = ctypes.c_char_p
            lib.moe_status_string.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _status_string(s: int) -> str:
    try:
        return load_library(build_if_missing=False).moe_status_string(s).decode()
    except Exception:  # the library itself may be what is missing
        return MOE_STATUS.get(s, f"status {s}")


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("the MoE layer runs on the GPU only: pass CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dims(d) -> Dims:
    return d if isinstance(d, Dims) else Dims(*[int(v) for v in d])


def _check(status: int, what: str):
    if status != 0:
        raise MoEError(status, what)


def moe_workspace_size(dims) -> int:
    return int(load_library().moe_workspace_size(ctypes.byref(_dims(dims))))


def moe_workspace_init(workspace: torch.Tensor, stream=None):
    _check(load_library().moe_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                             _stream(stream)), "moe_workspace_init")


def new_workspace(dims, device="cuda") -> torch.Tensor:
    """A zero-filled uint8 device workspace of moe_workspace_size(dims) bytes."""
    n = moe_workspace_size(dims)
    if n == 0:
        raise MoEError(2, "moe_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def moe_route(dims, x, weights: Weights, ids, topk_w, counts, offsets, perm, workspace, stream=None):
    w = weights.to_c()
    _check(load_library().moe_route(ctypes.byref(_dims(dims)), _ptr(x), ctypes.byref(w), _ptr(ids), _ptr(topk_w),
                                    _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream)), "moe_route")


def moe_route_noalloc(dims, x, weights: Weights, ids, topk_w, counts, offsets, perm, stream=None):
    """moe_route without a workspace (for callers that cannot allocate device memory)."""
    w = weights.to_c()
    _check(load_library().moe_route_noalloc(ctypes.byref(_dims(dims)), _ptr(x), ctypes.byref(w), _ptr(ids),
                                            _ptr(topk_w), _ptr(counts), _ptr(offsets), _ptr(perm), _stream(stream)),
           "moe_route_noalloc")


def moe_router_stats(dims, x, weights: Weights, P, f, loss, workspace, stream=None):
    """Load-balancing statistics: P [E] and f [E] fp32 (mean router probability, share of the
    assignments) and loss [1] fp32 = 0.001 * E * sum(f * P)."""
    w = weights.to_c()
    _check(load_library().moe_router_stats(ctypes.byref(_dims(dims)), _ptr(x), ctypes.byref(w), _ptr(P), _ptr(f),
                                           _ptr(loss), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _stream(stream)), "moe_router_stats")


def moe_forward(dims, x, weights: Weights, residual, out, workspace, stream=None):
    w = weights.to_c()
    _check(load_library().moe_forward(ctypes.byref(_dims(dims)), _ptr(x), ctypes.byref(w), _ptr(residual), _ptr(out),
                                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(stream)), "moe_forward")


def _ptr_host(t) -> int:
    """Address of a pinned (page-locked) host tensor, for the host-resident expert weights."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if t.is_cuda or not t.is_pinned():
        raise ValueError("host-resident expert weights must be pinned CPU tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def moe_expert_shadow_size(dims) -> int:
    return int(load_library().moe_expert_shadow_size(ctypes.byref(_dims(dims))))


def moe_forward_host_experts(dims, x, weights: Weights, residual, out, shadow, workspace, stream=None):
    """moe_forward with weights.gate_up and weights.down in pinned host memory: the experts
    each call touches are copied over the host link into `shadow` (a uint8 CUDA tensor of
    moe_expert_shadow_size(dims) bytes) and run from there."""
    w = CWeights(*[(_ptr_host(getattr(weights, f.name)) if f.name in ("gate_up", "down") else _ptr(getattr(weights, f.name)))
                   for f in fields(weights)])
    _check(load_library().moe_forward_host_experts(ctypes.byref(_dims(dims)), _ptr(x), ctypes.byref(w), _ptr(residual),
                                                   _ptr(out), _ptr(shadow), shadow.numel() * shadow.element_size(),
                                                   _ptr(workspace), workspace.numel() * workspace.element_size(),
                                                   _stream(stream)), "moe_forward_host_experts")


def _ptr_cpu(t, nbytes: int) -> int | None:
    """Address of a contiguous CPU tensor (pinned or pageable) of at least nbytes bytes."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if t.is_cuda:
        raise ValueError("host-side token rows must be CPU tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    if t.numel() * t.element_size() < nbytes:
        raise ValueError(f"host tensor holds {t.numel() * t.element_size()} bytes, the layer needs {nbytes}")
    return t.data_ptr()


def moe_forward_host_io(dims, x, weights: Weights, residual, out, x_dev, out_dev, workspace, stream=None):
    """moe_forward with the token rows in host memory: x (and residual, when given) are CPU
    tensors copied into the device staging tensors x_dev (and out_dev), the layer runs, and
    out_dev is copied back into the CPU tensor out, all in order on `stream`. Pinned host
    tensors keep the copies asynchronous (and one token, with x, residual and out pinned, runs
    in one kernel that reads and writes them over the host link, with no copy); out holds the
    result once the stream has passed the call."""
    d = _dims(dims)
    nbytes = d.T * d.H * 2
    for t in (x_dev, out_dev):
        if t is not None and t.numel() * t.element_size() < nbytes:
            raise ValueError("device staging tensors must hold [T, H] bf16")
    _check(load_library().moe_forward_host_io(ctypes.byref(d), _ptr_cpu(x, nbytes), ctypes.byref(weights.to_c()),
                                              _ptr_cpu(residual, nbytes), _ptr_cpu(out, nbytes), _ptr(x_dev),
                                              _ptr(out_dev), _ptr(workspace),
                                              workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_forward_host_io")


class ForwardHostIO:
    """moe_forward_host_io with everything but the host buffers marshalled once.

    A decode loop calls the same layer with the same weights, staging tensors and workspace
    on every step; this object converts those (and the stream, the current one when none is
    given) into C arguments at construction and keeps references to the tensors, so each
    call only checks and passes the host tensors. The tensors must not be resized or
    re-pointed (``set_``) while the object is in use."""

    def __init__(self, dims, weights: Weights, x_dev, out_dev, workspace, stream=None):
        self._d = _dims(dims)
        self._nbytes = self._d.T * self._d.H * 2
        for t in (x_dev, out_dev):
            if t is not None and t.numel() * t.element_size() < self._nbytes:
                raise ValueError("device staging tensors must hold [T, H] bf16")
        self._w = weights.to_c()
        self._keep = (weights, x_dev, out_dev, workspace)
        self._fixed = (ctypes.byref(self._d), ctypes.byref(self._w))
        self._staging = (_ptr(x_dev), _ptr(out_dev), _ptr(workspace), workspace.numel() * workspace.element_size(),
                         _stream(stream))
        self._fn = load_library().moe_forward_host_io

    def __call__(self, x, out, residual=None):
        n = self._nbytes
        _check(self._fn(self._fixed[0], _ptr_cpu(x, n), self._fixed[1], _ptr_cpu(residual, n), _ptr_cpu(out, n),
                        *self._staging), "moe_forward_host_io")


def moe_rmsnorm(dims, x, gamma, eps: float, xn, stream=None):
    _check(load_library().moe_rmsnorm(ctypes.byref(_dims(dims)), _ptr(x), _ptr(gamma), float(eps), _ptr(xn),
                                      _stream(stream)), "moe_rmsnorm")


def moe_last_device_error(workspace, stream=None) -> int:
    """Synchronise and return (and clear) the device error status kept in the workspace."""
    return int(load_library().moe_last_device_error(_ptr(workspace), _stream(stream)))


def moe_set_trace(kernel, start_events=(), stop_events=()):
    """Record the given torch.cuda.Event pairs around every launch of ``kernel`` (a name of
    KERNELS or its id), cycling through them; empty sequences clear the trace."""
    kid = KERNELS[kernel] if isinstance(kernel, str) else int(kernel)
    n = len(start_events)
    if n != len(stop_events):
        raise ValueError("start and stop event lists differ in length")
    arr = ctypes.c_void_p * max(n, 1)
    st = arr(*[e.cuda_event for e in start_events]) if n else None
    sp = arr(*[e.cuda_event for e in stop_events]) if n else None
    _check(load_library().moe_set_trace(kid, st, sp, n), "moe_set_trace")


def moe_test_set_wait(wait_ns: int = 0, suppress: int = 0):
    """Testing aid: time limit (ns, 0 = the default of ~1 s) of the bounded device waits of the
    one-token and streaming kernels, and a signal to hold back (TEST_SUPPRESS_*) so that a wait
    runs out; moe_test_set_wait() restores normal operation."""
    _check(load_library().moe_test_set_wait(int(wait_ns), int(suppress)), "moe_test_set_wait")


def moe_launch_count() -> int:
    return int(load_library().moe_launch_count())


def moe_workspace_tap(dims, tap: int) -> tuple[int, int]:
    off, nb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load_library().moe_workspace_tap(ctypes.byref(_dims(dims)), int(tap), ctypes.byref(off), ctypes.byref(nb)),
           "moe_workspace_tap")
    return off.value, nb.value
