"""moe_route_noalloc: the routing entry point for callers that cannot allocate device memory.

Its scratch is a fixed array inside the library instead of a caller-provided workspace. This
file is named so that pytest collects it last. It calls the entry point through the C ABI,
twice in a row on two inputs whose routings differ (the second call must not see the first
call's leftovers), on token counts from 1 to the largest supported (64), on the full layer
shape and the tiny one (E = 32, K = 4), with and without a router bias and with the bf16-typed
scores, and compares each result with moe_route's and with the oracle's: expert ids, counts,
offsets and dispatch permutation bit for bit, routing weights within the routing-weight
tolerance of the other GPU tests. It also checks the size limit."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
import sparse_moe_ffn_router_gb300 as moe
from sparse_moe_ffn_router_gb300.binding import CWeights, Dims
from tests.gpu_helpers import W_TOL, Layer, run_route
from tests.inputs import exact_score_inputs

pytestmark = pytest.mark.gpu


def _entry():
    lib = moe.load_library()
    fn = lib.moe_route_noalloc
    P = ctypes.c_void_p
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(Dims), P, ctypes.POINTER(CWeights), P, P, P, P, P, P]
    return fn


def _call(fn, dims, x, W):
    T, H, E, K = dims[:4]
    dev = x.device
    out = dict(ids=torch.full((T, K), -1, dtype=torch.int32, device=dev),
               w=torch.full((T, K), -1.0, dtype=torch.float32, device=dev),
               counts=torch.full((E,), -1, dtype=torch.int32, device=dev),
               offsets=torch.full((E + 1,), -1, dtype=torch.int32, device=dev),
               perm=torch.full((T * K,), -1, dtype=torch.int32, device=dev))
    cw = W.to_c()
    st = fn(ctypes.byref(Dims(*dims)), x.data_ptr(), ctypes.byref(cw), out["ids"].data_ptr(), out["w"].data_ptr(),
            out["counts"].data_ptr(), out["offsets"].data_ptr(), out["perm"].data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st, {k: v.cpu().numpy() for k, v in out.items()}


def _same(got, ref, what, w_tol=W_TOL):
    for k in ("ids", "counts", "offsets", "perm"):
        assert np.array_equal(got[k], ref[k]), f"{what}: {k}"
    np.testing.assert_allclose(got["w"], ref["w"], rtol=0, atol=w_tol, err_msg=f"{what}: routing weights")


CASES = [  # (dims, Zipf exponent of the router bias or None)
    ((1, 2048, 256, 8, 512, 512), None),
    ((7, 2048, 256, 8, 512, 512), None),
    ((33, 2048, 256, 8, 512, 512), None),
    ((64, 2048, 256, 8, 512, 512), None),
    ((8, 512, 32, 4, 128, 128), None),
    ((33, 2048, 256, 8, 512, 512), 1.1),
]


@pytest.mark.parametrize("dims,zipf", CASES, ids=lambda c: "x".join(map(str, c)) if isinstance(c, tuple) else f"zipf{c}")
def test_route_noalloc_matches_moe_route_and_the_oracle_twice(dims, zipf):
    fn = _entry()
    # two inputs whose routings differ: the second call must keep nothing of the first
    for seed in (2024, 2025):
        L = Layer(dims, seed=seed + dims[0], zipf_s=zipf)
        st, got = _call(fn, dims, L.xd, L.W)
        assert st == 0, moe.binding._status_string(st)
        _same(got, run_route(dims, L.xd, L.W), f"{dims} seed {seed}: against moe_route")
        _same(got, oracle.route(dims, L.x, L.router_w, L.router_b), f"{dims} seed {seed}: against the oracle")


def test_route_noalloc_bf16_scores_twice():
    """The bf16-typed scores (MOE_FLAG_BF16_SCORES) with a router bias, on inputs whose fp32
    scores are exact in any summation order, so that the roundings and their ties agree with
    the oracle's bit for bit."""
    fn = _entry()
    base = (33, 2048, 256, 8, 512, 512)
    dims = base + (moe.FLAG_BF16_SCORES,)
    for seed in (31, 32):
        r = exact_score_inputs(base, seed, with_bias=True)
        W = Layer(base, seed=seed, gap=False)
        W.W.router_w, W.W.shared_gate, W.W.router_b = r["router_w"].cuda(), r["shared_gate"].cuda(), r["router_b"].cuda()
        xd = r["x"].cuda()
        st, got = _call(fn, dims, xd, W.W)
        assert st == 0, moe.binding._status_string(st)
        _same(got, run_route(dims, xd, W.W), f"seed {seed}: against moe_route", w_tol=1e-5)
        _same(got, oracle.route(dims, r["x"], r["router_w"], r["router_b"]), f"seed {seed}: against the oracle",
              w_tol=1e-5)


def test_route_noalloc_rejects_sizes_beyond_its_scratch():
    fn = _entry()
    dims = (65, 2048, 256, 8, 512, 512)  # more tokens than the fixed scratch holds
    x = torch.zeros(65, 2048, dtype=torch.bfloat16, device="cuda")
    W = Layer((1, 2048, 256, 8, 512, 512), seed=1, gap=False).W
    st, _ = _call(fn, dims, x, W)
    assert st == 2  # MOE_ERR_UNSUPPORTED_SHAPE
