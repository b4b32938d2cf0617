"""Routed experts resident in host memory (moe_forward_host_experts): gate_up and down in
pinned, device-mapped host memory, the touched experts copied over the host link into a
device shadow after the routing, the layer run from there. Compared with the oracle on the
regimes the entry point uses (one-cluster routing + streaming experts for a few tokens, the
split router + streaming experts, the tensor-core GEMMs), and bit for bit with moe_forward on
device-resident weights where both take the same kernels."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
import sparse_moe_ffn_router_gb300 as moe
from sparse_moe_ffn_router_gb300 import binding, synth
from tests.gpu_helpers import assert_close
from tests.inputs import gap_controlled_x

pytestmark = pytest.mark.gpu


def _layer(dims, seed, layer=0):
    T, H, E, K, I, Is = dims
    w = synth.make_weights(H, E, I, Is, seed, layer)
    x, _ = gap_controlled_x(dims, w["router_w"], w["router_b"], seed, layer)
    dev = {k: (None if v is None else v.cuda()) for k, v in w.items()}
    host = dict(dev)
    host["gate_up"] = w["gate_up"].pin_memory()
    host["down"] = w["down"].pin_memory()
    return x, w, moe.Weights.from_dict(dev), moe.Weights.from_dict(host)


def _run_host(dims, xd, Wh, shadow=None, ws=None):
    T, H = dims[:2]
    shadow = torch.zeros(moe.moe_expert_shadow_size(dims), dtype=torch.uint8, device="cuda") if shadow is None else shadow
    ws = moe.new_workspace(dims, xd.device) if ws is None else ws
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward_host_experts(dims, xd, Wh, None, out, shadow, ws)
    torch.cuda.synchronize()
    assert moe.moe_last_device_error(ws) == 0
    return out, shadow


def _run_device(dims, xd, Wd):
    T, H = dims[:2]
    ws = moe.new_workspace(dims, xd.device)
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(dims, xd, Wd, None, out, ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dims", [(1, 2048, 256, 8, 512, 512), (5, 2048, 256, 8, 512, 512),
                                  (64, 2048, 256, 8, 512, 512), (300, 512, 32, 4, 128, 128)],
                         ids=lambda d: "x".join(map(str, d)))
def test_host_experts_parity(dims):
    x, w, Wd, Wh = _layer(dims, 61 + dims[0])
    out, _ = _run_host(dims, x.cuda(), Wh)
    ref = oracle.forward(dims, x, w)
    assert_close(out.float().cpu().numpy(), ref["out"], f"moe_forward_host_experts {dims}")
    if dims[0] > 8:  # same kernels as moe_forward, only the weights' home differs
        assert torch.equal(out, _run_device(dims, x.cuda(), Wd))


def test_one_shadow_serves_layers_in_turn():
    dims = (64, 2048, 256, 8, 512, 512)
    xa, wa, Wda, Wha = _layer(dims, 3, 0)
    xb, wb, Wdb, Whb = _layer(dims, 3, 1)
    out_a, shadow = _run_host(dims, xa.cuda(), Wha)
    out_b, _ = _run_host(dims, xb.cuda(), Whb, shadow=shadow)
    out_a2, _ = _run_host(dims, xa.cuda(), Wha, shadow=shadow)
    assert torch.equal(out_a, out_a2)
    assert torch.equal(out_b, _run_device(dims, xb.cuda(), Wdb))


def test_device_pointers_are_refused_as_host_experts():
    dims = (8, 2048, 256, 8, 512, 512)
    x, w, Wd, Wh = _layer(dims, 9)
    lib = binding.load_library()
    d = binding.Dims(*dims)
    cw = Wd.to_c()  # gate_up and down in device memory: not host-mapped memory
    ws = moe.new_workspace(dims)
    shadow = torch.empty(moe.moe_expert_shadow_size(dims), dtype=torch.uint8, device="cuda")
    out = torch.empty(8, 2048, dtype=torch.bfloat16, device="cuda")
    st = lib.moe_forward_host_experts(ctypes.byref(d), x.cuda().data_ptr(), ctypes.byref(cw), None, out.data_ptr(),
                                      shadow.data_ptr(), shadow.numel(), ws.data_ptr(), ws.numel(), None)
    assert st == 1
    with pytest.raises(ValueError, match="pinned"):
        moe.moe_forward_host_experts(dims, x.cuda(), Wd, None, out, shadow, ws)


def test_mapping_smaller_than_the_expert_tensors_is_rejected():
    """The fetch kernel may read any expert's rows, so the registered host allocation holding
    gate_up must cover the whole [E, 2I, H] tensor: a buffer of which only the first half is
    registered (and mapped) is refused on the host before anything runs. (A router bias keeps
    the routing on experts 0..K-1, whose rows lie in the registered half, so even a call that
    slipped through would read registered memory only.)"""
    dims = (8, 512, 32, 4, 128, 128)
    x, w, _, Wh = _layer(dims, seed=41)
    bias = torch.zeros(dims[2], dtype=torch.bfloat16)
    bias[: dims[3]] = 100.0
    gu = w["gate_up"].clone()  # pageable; half of it registered below
    half = gu.numel() * gu.element_size() // 2
    assert dims[3] * 2 * dims[4] * dims[1] * 2 <= half  # the routed experts' rows are in the registered half
    cudart = torch.cuda.cudart()
    assert int(cudart.cudaHostRegister(gu.data_ptr(), half, 2)) == 0  # cudaHostRegisterMapped
    try:
        bad = moe.Weights(Wh.router_w, bias.cuda(), gu, Wh.down, Wh.shared_gate_up, Wh.shared_down, Wh.shared_gate)
        with pytest.raises(binding.MoEError) as e:
            _run_host(dims, x.cuda(), bad)
        assert e.value.status == 1  # MOE_ERR_INVALID_ARG
    finally:
        torch.cuda.synchronize()
        cudart.cudaHostUnregister(gu.data_ptr())
