"""Test-side input preparation: seeded layers whose routing is unambiguous.

The router's K-th and (K+1)-th scores, and every adjacent pair among the top K+1, are kept
at least GAP apart (measured on the oracle's fp64 logits, bias included) by redrawing the
offending token rows from the next stream of the seeded generator. With that gap, fp32
scoring on the GPU and fp64 scoring in the oracle must agree on the experts and on their
slot order, so routing can be compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from sparse_moe_ffn_router_gb300 import synth
from sparse_moe_ffn_router_gb300.workloads import Workload

GAP = 1e-3
MAX_ATTEMPTS = 64


def top_gaps(logits: np.ndarray, K: int) -> np.ndarray:
    """Smallest adjacent gap among the top K+1 scores of each row ([T])."""
    E = logits.shape[1]
    k1 = min(K + 1, E)
    top = -np.sort(-logits, axis=1)[:, :k1]
    if k1 < 2:
        return np.full(logits.shape[0], np.inf)
    return np.min(top[:, :-1] - top[:, 1:], axis=1)


def gap_controlled_x(dims, router_w, router_b, seed: int, layer: int = 0, device="cpu"):
    """x [T,H] bf16 whose rows all have routing gaps >= GAP. Returns (x, attempts)."""
    T, H, E, K = dims[0], dims[1], dims[2], dims[3]
    attempts = np.zeros(T, np.int64)
    x = synth.make_x(T, H, seed, layer)
    for _ in range(MAX_ATTEMPTS):
        lg = oracle.router_logits(dims, x, router_w, router_b)
        bad = np.nonzero(top_gaps(lg, K) < GAP)[0]
        if bad.size == 0:
            return x.to(device), attempts
        attempts[bad] += 1
        x = synth.make_x(T, H, seed, layer, attempts=attempts)
    raise RuntimeError("could not separate the routing scores")


def layer_inputs(wl: Workload, device="cpu", layer: int = 0, gap=True):
    """(weights dict, x) of one layer of a workload, generated on ``device``."""
    w = synth.make_weights(wl.H, wl.E, wl.I, wl.Is, wl.seed, layer, wl.zipf_s, device=device)
    if gap:
        x, _ = gap_controlled_x(wl.dims, w["router_w"], w["router_b"], wl.seed, layer, device=device)
    else:
        x = synth.make_x(wl.T, wl.H, wl.seed, layer, device=device)
    return w, x


def to_host(w: dict) -> dict:
    return {k: (None if v is None else v.detach().cpu()) for k, v in w.items()}


def bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def exact_score_inputs(dims, seed: int, with_bias: bool = False, layer: int = 0) -> dict:
    """Router inputs whose fp32 scores are exact in any summation order, for comparing the
    bf16-typed scores bit for bit: x in {-1, 0, 1}; router and shared-gate weights integer
    multiples of 2^-7 up to 40/128 (6 significant bits, exact in bf16); the bias (when asked)
    a multiple of 2^-5 up to 3 (7 bits). Every score is then an integer multiple of 2^-7 below
    2^17 * 2^-7, exact in fp32 whatever the order of the additions, and mostly needs more than
    bf16's 8 significant bits, so the rounding and its ties are exercised. Drawn from the
    seeded synthetic streams (N(0, 1) token values and N(0, 16^2) weights, clamped and
    rounded)."""
    T, H, E = dims[:3]
    z = synth.make_x(T, H, seed, layer, tag="x_exact").float()
    x = torch.round(torch.clamp(z, -1.4, 1.4)).to(torch.bfloat16)
    wr = synth.normal_bf16((E, H), 16.0, synth.stream_key(seed, layer, "router_w_exact")).float()
    wr = (torch.round(torch.clamp(wr, -40, 40)) / 128).to(torch.bfloat16)
    sg = synth.normal_bf16((1, H), 16.0, synth.stream_key(seed, layer, "shared_gate_exact")).float()
    sg = (torch.round(torch.clamp(sg, -40, 40)) / 128).to(torch.bfloat16)
    br = None
    if with_bias:
        b = synth.normal_bf16((E,), 1.0, synth.stream_key(seed, layer, "router_b_exact")).float()
        br = (torch.round(torch.clamp(b, -3, 3) * 32) / 32).to(torch.bfloat16)
    return dict(x=x, router_w=wr, shared_gate=sg, router_b=br)
