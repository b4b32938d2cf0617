"""moe_route_noalloc: the routing entry point for callers that cannot allocate device memory.

Its scratch is a fixed array inside the library instead of a caller-provided workspace. This
file is named so that pytest collects it last. It calls the entry point through the C ABI on
the full layer shape at the largest supported token count, twice in a row (the second call
must not see the first call's leftovers), and compares each result with moe_route's: expert
ids, counts, offsets and dispatch permutation bit for bit, routing weights within the
routing-weight tolerance of the other GPU tests. It also checks the size limit."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import sparse_moe_ffn_router_gb300 as moe
from sparse_moe_ffn_router_gb300.binding import CWeights, Dims
from tests.gpu_helpers import W_TOL, Layer, run_route

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


def test_route_noalloc_matches_moe_route_twice():
    fn = _entry()
    dims = (64, 2048, 256, 8, 512, 512)
    L = Layer(dims, seed=2024)
    ref = run_route(dims, L.xd, L.W)
    # a second input whose routing differs, to show the second call keeps nothing stale
    L2 = Layer(dims, seed=2025)
    ref2 = run_route(dims, L2.xd, L2.W)
    for lay, r in ((L, ref), (L2, ref2)):
        st, got = _call(fn, dims, lay.xd, lay.W)
        assert st == 0, moe.binding._status_string(st)
        for k in ("ids", "counts", "offsets", "perm"):
            assert np.array_equal(got[k], r[k]), k
        np.testing.assert_allclose(got["w"], r["w"], rtol=0, atol=W_TOL)


def test_route_noalloc_rejects_sizes_beyond_its_scratch():
    fn = _entry()
    dims = (65, 2048, 256, 8, 512, 512)  # more tokens than the fixed scratch holds
    x = torch.zeros(65, 2048, dtype=torch.bfloat16, device="cuda")
    W = Layer((1, 2048, 256, 8, 512, 512), seed=1, gap=False).W
    st, _ = _call(fn, dims, x, W)
    assert st == 2  # MOE_ERR_UNSUPPORTED_SHAPE
