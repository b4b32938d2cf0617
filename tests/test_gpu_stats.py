"""Load-balancing statistics (moe_router_stats, called through the C ABI) against the oracle:
per-expert mean router probability P, assignment share f and the auxiliary loss
0.001 * E * sum(f * P), on every workload shape and on edge shapes.

Tolerances: the GPU scores are fp32 sums of bf16 products (score error ~1e-4 on these
inputs, as derived for the routing weights in gpu_helpers), so each softmax probability is
off by a relative ~2e-4 at most and so is its mean over the tokens; P and the loss are
compared within a relative 1e-3. The assignment counts f * T * K must match exactly (routing
is bit-exact on gap-controlled inputs), and repeated calls must agree bit for bit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import sparse_moe_ffn_router_gb300 as moe
from sparse_moe_ffn_router_gb300.workloads import WORKLOADS
from tests.gpu_helpers import Layer

pytestmark = pytest.mark.gpu

P_RTOL, P_ATOL = 1e-3, 1e-7


def run_stats(dims, xd, W, ws=None):
    E = dims[2]
    ws = moe.new_workspace(dims, xd.device) if ws is None else ws
    P = torch.full((E,), -1.0, dtype=torch.float32, device=xd.device)
    f = torch.full((E,), -1.0, dtype=torch.float32, device=xd.device)
    loss = torch.full((4,), -1.0, dtype=torch.float32, device=xd.device)
    moe.moe_router_stats(dims, xd, W, P, f, loss, ws)
    torch.cuda.synchronize()
    assert moe.moe_last_device_error(ws) == 0
    return P.cpu().numpy(), f.cpu().numpy(), float(loss[0].item()), ws


def check_stats(L: Layer):
    T, K = L.T, L.K
    ref = oracle.router_stats(L.dims, L.x, L.router_w, L.router_b)
    P, f, loss, ws = run_stats(L.dims, L.xd, L.W)
    np.testing.assert_allclose(P, ref["P"], rtol=P_RTOL, atol=P_ATOL)
    counts = np.rint(f.astype(np.float64) * T * K).astype(np.int64)
    np.testing.assert_array_equal(counts, np.rint(ref["f"] * T * K).astype(np.int64))
    np.testing.assert_allclose(f, ref["f"], rtol=1e-6)
    assert loss == pytest.approx(ref["loss"], rel=P_RTOL)
    P2, f2, loss2, _ = run_stats(L.dims, L.xd, L.W, ws)
    assert np.array_equal(P, P2) and np.array_equal(f, f2) and loss == loss2


@pytest.mark.parametrize("name", ["tiny_T8", "decode_T1", "decode_T64", "prefill_T4096_zipf"])
def test_router_stats_parity(name):
    wl = WORKLOADS[name]
    check_stats(Layer(wl.dims, wl.seed, wl.zipf_s))


@pytest.mark.parametrize("dims", [(1, 128, 8, 1, 64, 64), (1, 128, 256, 2, 64, 64), (67, 256, 8, 8, 64, 128),
                                  (300, 384, 40, 3, 192, 64)],
                         ids=lambda d: "x".join(map(str, d)))
def test_router_stats_edge_shapes(dims):
    check_stats(Layer(dims, seed=200 + dims[0], router_std=0.1))


def test_router_stats_uniform_scores_and_zero_tokens():
    dims = (16, 256, 32, 4, 64, 64)
    L = Layer(dims, seed=7, gap=False)
    P, f, loss, _ = run_stats(dims, torch.zeros_like(L.xd), L.W)  # every score 0
    np.testing.assert_array_equal(P, np.full(32, 1.0 / 32, np.float32))
    np.testing.assert_array_equal(f, np.r_[np.full(4, 0.25), np.zeros(28)].astype(np.float32))
    assert loss == pytest.approx(0.001, rel=1e-6)
    z = (0,) + dims[1:]
    P, f, loss, _ = run_stats(z, torch.empty(0, 256, dtype=torch.bfloat16, device="cuda"), L.W)
    assert not P.any() and not f.any() and loss == 0.0
