"""The oracle: a plain, slow fp64 CPU model of the sparse MoE feed-forward layer.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA library of the product
path (``sparse_moe_ffn_router_gb300``), and that package never imports it.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64, OpenMP over tokens). This module
only compiles it with gcc and marshals numpy arrays through ctypes. bf16 tensors are passed
as ``uint16`` arrays holding the raw bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


# dims tuples are (T, H, E, K, I, Is) or (T, H, E, K, I, Is, flags)
BF16_SCORES = 1  # router and shared-gate scores typed bf16 (rounded before ranking and sigmoid)


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("K", ctypes.c_int32), ("I", ctypes.c_int32), ("Is", ctypes.c_int32), ("flags", ctypes.c_int32)]


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared library (gcc, -O2, OpenMP when available)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.oracle_router_logits.argtypes = [ctypes.POINTER(Dims), P, P, P, P]
            lib.oracle_route.restype = ctypes.c_int
            lib.oracle_route.argtypes = [ctypes.POINTER(Dims)] + [P] * 10
            lib.oracle_permute.argtypes = [ctypes.POINTER(Dims)] + [P] * 5
            lib.oracle_forward.restype = ctypes.c_int
            lib.oracle_forward.argtypes = [ctypes.POINTER(Dims)] + [P] * 16
            lib.oracle_rmsnorm.argtypes = [ctypes.c_int32, ctypes.c_int32, P, P, ctypes.c_double, P]
            lib.oracle_router_stats.argtypes = [ctypes.POINTER(Dims)] + [P] * 6
            _lib = lib
    return _lib


def _u16(a, shape=None):
    """A C-contiguous uint16 view of a bf16 bit-pattern array (numpy or torch)."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # a torch tensor: copy its bits to host
        import torch
        a = a.detach().contiguous().cpu()
        if a.dtype == torch.bfloat16:
            a = a.view(torch.int16)
        a = a.numpy()
    a = np.ascontiguousarray(a).view(np.uint16)
    if shape is not None:
        a = a.reshape(shape)
    return a


def _p(a):
    return None if a is None else a.ctypes.data


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def round_bf16(v: float) -> int:
    return int(_load().oracle_round_bf16(float(v)))


def router_logits(dims, x, router_w, router_b=None) -> np.ndarray:
    lib = _load()
    d = Dims(*dims)
    x, wr, br = _u16(x), _u16(router_w), _u16(router_b)
    out = np.empty((d.T, d.E), np.float64)
    lib.oracle_router_logits(ctypes.byref(d), _p(x), _p(wr), _p(br), _p(out))
    return out


def route(dims, x, router_w, router_b=None, want_probs=False) -> dict:
    """Routing of every token: ids [T,K] i32 (slot order), w [T,K] f64, counts [E],
    offsets [E+1], perm [T*K], inv [T*K] (and probs [T,E] when asked)."""
    lib = _load()
    d = Dims(*dims)
    T, E, K = d.T, d.E, d.K
    x, wr, br = _u16(x), _u16(router_w), _u16(router_b)
    r = dict(ids=np.zeros((T, K), np.int32), w=np.zeros((T, K), np.float64),
             counts=np.zeros(E, np.int32), offsets=np.zeros(E + 1, np.int32),
             perm=np.zeros(T * K, np.int32), inv=np.zeros(T * K, np.int32))
    probs = np.zeros((T, E), np.float64) if want_probs else None
    rc = lib.oracle_route(ctypes.byref(d), _p(x), _p(wr), _p(br), _p(r["ids"]), _p(r["w"]), _p(probs),
                          _p(r["counts"]), _p(r["offsets"]), _p(r["perm"]), _p(r["inv"]))
    if rc != 0:
        raise ValueError(f"oracle_route rejected dims {dims}")
    if want_probs:
        r["probs"] = probs
    return r


def router_stats(dims, x, router_w, router_b=None) -> dict:
    """Load-balancing statistics: P [E] (mean router probability), f [E] (share of the
    (token, slot) assignments) and loss = 0.001 * E * sum(f * P), all fp64."""
    lib = _load()
    d = Dims(*dims)
    x, wr, br = _u16(x), _u16(router_w), _u16(router_b)
    P = np.zeros(d.E, np.float64)
    f = np.zeros(d.E, np.float64)
    loss = np.zeros(1, np.float64)
    if lib.oracle_router_stats(ctypes.byref(d), _p(x), _p(wr), _p(br), _p(P), _p(f), _p(loss)) != 0:
        raise ValueError(f"oracle_router_stats rejected dims {dims}")
    return dict(P=P, f=f, loss=float(loss[0]))


def permute(dims, ids) -> dict:
    lib = _load()
    d = Dims(*dims)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    r = dict(counts=np.zeros(d.E, np.int32), offsets=np.zeros(d.E + 1, np.int32),
             perm=np.zeros(d.T * d.K, np.int32), inv=np.zeros(d.T * d.K, np.int32))
    lib.oracle_permute(ctypes.byref(d), _p(ids), _p(r["counts"]), _p(r["offsets"]), _p(r["perm"]), _p(r["inv"]))
    return r


def forward(dims, x, w, residual=None, taps=False) -> dict:
    """The layer output out [T,H] f64 (= residual + MoE(x), or MoE(x) when residual is None).

    ``w`` maps names to bf16 tensors: router_w [E,H], router_b [E] or None, gate_up [E,2I,H],
    down [E,H,I], shared_gate_up [2Is,H], shared_down [H,Is], shared_gate [1,H].
    With ``taps`` the per-slot h [T,K,I], y [T,K,H], shared ys [T,H], gate sg [T], ids, w."""
    lib = _load()
    d = Dims(*dims)
    T, H, K, I = d.T, d.H, d.K, d.I
    arrs = [_u16(x), _u16(w["router_w"]), _u16(w.get("router_b")), _u16(w["gate_up"]), _u16(w["down"]),
            _u16(w["shared_gate_up"]), _u16(w["shared_down"]), _u16(w["shared_gate"]), _u16(residual)]
    out = np.zeros((T, H), np.float64)
    t = {}
    if taps:
        t = dict(h=np.zeros((T, K, I)), y=np.zeros((T, K, H)), ys=np.zeros((T, H)), sg=np.zeros(T),
                 ids=np.zeros((T, K), np.int32), w=np.zeros((T, K)))
    rc = lib.oracle_forward(ctypes.byref(d), *[_p(a) for a in arrs], _p(out), _p(t.get("h")), _p(t.get("y")),
                            _p(t.get("ys")), _p(t.get("sg")), _p(t.get("ids")), _p(t.get("w")))
    if rc != 0:
        raise ValueError(f"oracle_forward rejected dims {dims}")
    t["out"] = out
    return t


def rmsnorm(x, gamma=None, eps=1e-6) -> np.ndarray:
    lib = _load()
    x = _u16(x)
    T, H = x.shape
    g = _u16(gamma)
    out = np.zeros((T, H), np.float64)
    lib.oracle_rmsnorm(T, H, _p(x), _p(g), float(eps), _p(out))
    return out


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round an fp64 array to bf16 (nearest, ties to even) with the oracle's own rounding."""
    lib = _load()
    flat = np.asarray(a, np.float64).ravel()
    out = np.fromiter((lib.oracle_round_bf16(float(v)) for v in flat), np.uint16, flat.size)
    return out.reshape(np.shape(a))


def bf16_bits_to_f64(a) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    a = _u16(a)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
