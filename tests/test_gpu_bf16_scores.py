"""bf16-typed router outputs (MOE_FLAG_BF16_SCORES) through the C ABI against the oracle's
same reading: every router score and the shared-gate score, bias included, rounded to bf16
before the softmax, the ranking and the sigmoid ("Qwen3.6 35B-A3B", Blocks: SparseMoe types
the router, the shared gate and `ranks` as T = bf16).

The router inputs come from tests.inputs.exact_score_inputs: x in {-1, 0, 1} and weights
that are small multiples of 2^-7, so every fp32 score on the GPU equals the oracle's fp64
score exactly, whatever the summation order. The bf16 roundings, and the many exact ties
they create, must then agree bit for bit: expert ids, counts, offsets and the dispatch
permutation are compared exactly on every routing regime (one-cluster router, small-T split
router, tensor-core GEMM router, the fused decode kernel and the workspace-free router). The
weights and gates are fp32 softmax / sigmoid of equal inputs: within 1e-5."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import sparse_moe_ffn_router_gb300 as moe
from sparse_moe_ffn_router_gb300 import synth
from tests.gpu_helpers import assert_close, read_tap, run_forward, run_route
from tests.inputs import exact_score_inputs

pytestmark = pytest.mark.gpu

F = moe.FLAG_BF16_SCORES
EXACT_TOL = 1e-5


def _layer(dims, seed, with_bias=False):
    T, H, E, K, I, Is = dims[:6]
    w = synth.make_weights(H, E, I, Is, seed)
    r = exact_score_inputs(dims, seed, with_bias)
    w["router_w"], w["shared_gate"], w["router_b"] = r["router_w"], r["shared_gate"], r["router_b"]
    wd = {k: (None if v is None else v.cuda()) for k, v in w.items()}
    return r["x"], w, r["x"].cuda(), moe.Weights.from_dict(wd)


def _shared_gate(dims, x, w):
    """sigmoid of the bf16-typed shared-gate score, from the oracle's scoring of that row."""
    T, H = dims[:2]
    z = oracle.router_logits((T, H, 1, 1, 64, 64, F), x, w["shared_gate"])[:, 0]
    return 1.0 / (1.0 + np.exp(-z))


def _check(gpu, ref, what):
    assert np.array_equal(gpu["ids"], ref["ids"]), f"{what}: expert ids differ"
    assert np.array_equal(gpu["counts"], ref["counts"]), f"{what}: counts differ"
    assert np.array_equal(gpu["offsets"], ref["offsets"]), f"{what}: offsets differ"
    assert np.array_equal(gpu["perm"], ref["perm"]), f"{what}: dispatch permutation differs"
    np.testing.assert_allclose(gpu["w"], ref["w"], rtol=0, atol=EXACT_TOL, err_msg=f"{what}: routing weights")


ROUTE_DIMS = [(8, 2048, 256, 8, 512, 512), (64, 2048, 256, 8, 512, 512), (200, 1024, 64, 6, 256, 256),
              (300, 2048, 256, 8, 512, 512), (4096, 2048, 256, 8, 512, 512)]


@pytest.mark.parametrize("dims", ROUTE_DIMS, ids=lambda d: "x".join(map(str, d)))
@pytest.mark.parametrize("with_bias", [False, True], ids=["nobias", "bias"])
def test_routing_is_bit_exact_with_bf16_scores(dims, with_bias):
    x, w, xd, W = _layer(dims, 31 + dims[0], with_bias)
    ref = oracle.route(dims + (F,), x, w["router_w"], w["router_b"])
    gpu = run_route(dims + (F,), xd, W)
    _check(gpu, ref, f"moe_route {dims}")
    if dims[0] >= 64:  # the inputs exercise the reading: bf16 scores change some routings
        plain = oracle.route(dims, x, w["router_w"], w["router_b"])
        assert (plain["ids"] != ref["ids"]).any()


def test_workspace_free_router_with_bf16_scores():
    dims = (48, 2048, 256, 8, 512, 512)
    x, w, xd, W = _layer(dims, 5, True)
    T, H, E, K = dims[:4]
    ref = oracle.route(dims + (F,), x, w["router_w"], w["router_b"])
    ids = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    tw = torch.zeros(T, K, dtype=torch.float32, device="cuda")
    counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    perm = torch.full((T * K,), -1, dtype=torch.int32, device="cuda")
    moe.moe_route_noalloc(dims + (F,), xd, W, ids, tw, counts, offsets, perm)
    torch.cuda.synchronize()
    gpu = dict(ids=ids.cpu().numpy(), w=tw.cpu().numpy(), counts=counts.cpu().numpy(),
               offsets=offsets.cpu().numpy(), perm=perm.cpu().numpy())
    _check(gpu, ref, "moe_route_noalloc")


FORWARD_DIMS = [(1, 2048, 256, 8, 512, 512), (5, 2048, 256, 8, 512, 512), (64, 2048, 256, 8, 512, 512),
                (300, 512, 32, 4, 128, 128)]


@pytest.mark.parametrize("dims", FORWARD_DIMS, ids=lambda d: "x".join(map(str, d)))
def test_forward_with_bf16_scores(dims):
    """Routing taps of moe_forward (the fused decode kernel for T <= 8) bit-exact, the shared
    gate from the rounded score, and the layer output within the layer tolerance."""
    T, H, E, K = dims[:4]
    x, w, xd, W = _layer(dims, 7 + dims[0], True)
    ref = oracle.forward(dims + (F,), x, w, taps=True)
    out, ws = run_forward(dims + (F,), xd, W)
    assert moe.moe_last_device_error(ws) == 0
    ids = read_tap(ws, dims, 3, torch.int32, (T, K)).cpu().numpy()
    tw = read_tap(ws, dims, 4, torch.float32, (T, K)).cpu().numpy()
    sg = read_tap(ws, dims, 2, torch.float32, (T,)).cpu().numpy()
    assert np.array_equal(ids, ref["ids"]), "expert ids differ"
    np.testing.assert_allclose(tw, ref["w"], rtol=0, atol=EXACT_TOL)
    np.testing.assert_allclose(sg, ref["sg"], rtol=EXACT_TOL, atol=0)
    np.testing.assert_allclose(sg, _shared_gate(dims, x, w), rtol=EXACT_TOL, atol=0)
    assert_close(out.float().cpu().numpy(), ref["out"], f"moe_forward {dims}")


@pytest.mark.parametrize("dims", [(64, 2048, 256, 8, 512, 512), (4096, 2048, 256, 8, 512, 512)],
                         ids=lambda d: "x".join(map(str, d)))
def test_router_stats_with_bf16_scores(dims):
    T, H, E, K = dims[:4]
    x, w, xd, W = _layer(dims, 3, True)
    ref = oracle.router_stats(dims + (F,), x, w["router_w"], w["router_b"])
    ws = moe.new_workspace(dims, xd.device)
    P = torch.empty(E, dtype=torch.float32, device="cuda")
    f = torch.empty(E, dtype=torch.float32, device="cuda")
    loss = torch.empty(4, dtype=torch.float32, device="cuda")
    moe.moe_router_stats(dims + (F,), xd, W, P, f, loss, ws)
    torch.cuda.synchronize()
    assert moe.moe_last_device_error(ws) == 0
    np.testing.assert_allclose(P.cpu().numpy(), ref["P"], rtol=1e-4, atol=1e-7)
    np.testing.assert_array_equal(np.rint(f.cpu().numpy().astype(np.float64) * T * K), np.rint(ref["f"] * T * K))
    assert float(loss[0]) == pytest.approx(ref["loss"], rel=1e-4)
