"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and compare it with
the oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_moe_ffn_router_gb300 as moe
from sparse_moe_ffn_router_gb300 import synth
from tests.inputs import gap_controlled_x

TOL_REL, TOL_ABS = 1e-2, 1e-3
# Renormalised routing weights (fp32 on the GPU, fp64 in the oracle). The GPU scores are fp32
# sums of H = 2048 bf16 products whose order differs between the CUDA-core and tensor-core
# paths; with sum|x_h w_h| ~ 26 on these inputs the score error is ~1e-4 (random-walk
# estimate sqrt(H) * 2^-24 * 26 * a few), and w_k = exp(l_k - l_0) / sum moves by at most
# about 2 * w_k * max|dl|. 5e-4 covers that and still fails a wrong renormalisation (errors of
# order 1e-1).
W_TOL = 5e-4


def tolerance(ref: np.ndarray) -> float:
    """max|gpu - oracle| <= 1e-2 * max|oracle| + 1e-3 (the layer's output bound)."""
    return TOL_REL * float(np.abs(ref).max()) + TOL_ABS


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str):
    err = float(np.abs(gpu.astype(np.float64) - ref).max()) if ref.size else 0.0
    tol = tolerance(ref) if ref.size else 0.0
    assert err <= tol, f"{what}: max|gpu-oracle| = {err:.3e} > {tol:.3e}"
    return err, tol


class Layer:
    """One layer's weights and a gap-controlled x, generated on the GPU; host copies of the
    router weights (and, lazily, of the experts) go to the oracle."""

    def __init__(self, dims, seed, zipf_s=None, layer=0, router_std=0.02, gap=True):
        self.dims = tuple(dims)
        T, H, E, K, I, Is = self.dims
        self.T, self.H, self.E, self.K, self.I, self.Is = self.dims
        dev = torch.device("cuda")
        self.wd = synth.make_weights(H, E, I, Is, seed, layer, zipf_s, device=dev, router_std=router_std)
        self.router_w = self.wd["router_w"].cpu()
        self.router_b = None if self.wd["router_b"] is None else self.wd["router_b"].cpu()
        if gap:
            x, _ = gap_controlled_x(self.dims, self.router_w, self.router_b, seed, layer)
        else:
            x = synth.make_x(T, H, seed, layer)
        self.x = x
        self.xd = x.to(dev)
        self.W = moe.Weights.from_dict(self.wd)
        self._host = None

    def host_weights(self) -> dict:
        if self._host is None:
            self._host = {k: (None if v is None else v.cpu()) for k, v in self.wd.items()}
        return self._host


def run_route(dims, xd, W, ws=None):
    T, H, E, K = dims[:4]
    dev = xd.device
    ws = moe.new_workspace(dims, dev) if ws is None else ws
    ids = torch.full((T, K), -1, dtype=torch.int32, device=dev)
    tw = torch.zeros(T, K, dtype=torch.float32, device=dev)
    counts = torch.full((E,), -1, dtype=torch.int32, device=dev)
    offsets = torch.full((E + 1,), -1, dtype=torch.int32, device=dev)
    perm = torch.full((T * K,), -1, dtype=torch.int32, device=dev)
    moe.moe_route(dims, xd, W, ids, tw, counts, offsets, perm, ws)
    torch.cuda.synchronize()
    assert moe.moe_last_device_error(ws) == 0
    return dict(ids=ids.cpu().numpy(), w=tw.cpu().numpy(), counts=counts.cpu().numpy(),
                offsets=offsets.cpu().numpy(), perm=perm.cpu().numpy())


def run_forward(dims, xd, W, residual=None, ws=None, out=None):
    T, H = dims[:2]
    ws = moe.new_workspace(dims, xd.device) if ws is None else ws
    out = torch.empty(T, H, dtype=torch.bfloat16, device=xd.device) if out is None else out
    moe.moe_forward(dims, xd, W, residual, out, ws)
    torch.cuda.synchronize()
    return out, ws


def read_tap(ws, dims, tap, dtype, shape):
    off, nb = moe.moe_workspace_tap(dims, tap)
    return ws[off:off + nb].view(dtype).view(*shape)


def check_routing(gpu: dict, ref: dict, what=""):
    assert np.array_equal(gpu["ids"], ref["ids"]), f"{what}: expert ids differ"
    assert np.array_equal(gpu["counts"], ref["counts"]), f"{what}: counts differ"
    assert np.array_equal(gpu["offsets"], ref["offsets"]), f"{what}: offsets differ"
    assert np.array_equal(gpu["perm"], ref["perm"]), f"{what}: dispatch permutation differs"
    np.testing.assert_allclose(gpu["w"], ref["w"], rtol=0, atol=W_TOL, err_msg=f"{what}: routing weights")
