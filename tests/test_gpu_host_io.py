"""The layer with its token rows in host memory (moe_forward_host_io): x and the residual are
copied from host buffers into device staging, the layer runs, and the output is copied back
(or, for one pinned token row, the one-token kernel reads and writes the host rows itself).
Compared with the oracle, and bit for bit with moe_forward on the same device inputs, in each
regime the entry point reaches (the fused one-token kernel, the streaming experts, the
tensor-core GEMMs), with pinned and pageable host buffers, with and without a residual, with
the output written over the host x, and through the prepared call (ForwardHostIO)."""
from __future__ import annotations

import ctypes

import pytest
import torch

import oracle
import sparse_moe_ffn_router_gb300 as moe
from sparse_moe_ffn_router_gb300 import binding, synth
from tests.gpu_helpers import assert_close
from tests.inputs import gap_controlled_x

pytestmark = pytest.mark.gpu

CASES = [(1, 2048, 256, 8, 512, 512), (64, 2048, 256, 8, 512, 512), (300, 512, 32, 4, 128, 128)]


def _layer(dims, seed):
    T, H, E, K, I, Is = dims
    w = synth.make_weights(H, E, I, Is, seed, 0)
    x, _ = gap_controlled_x(dims, w["router_w"], w["router_b"], seed, 0)
    residual = synth.normal_bf16((T, H), 1.0, synth.stream_key(seed, 1, "x"))
    W = moe.Weights.from_dict({k: (None if v is None else v.cuda()) for k, v in w.items()})
    return x, residual, w, W


def _device_forward(dims, x, residual, W):
    T, H = dims[:2]
    ws = moe.new_workspace(dims)
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(dims, x.cuda(), W, None if residual is None else residual.cuda(), out, ws)
    torch.cuda.synchronize()
    return out.cpu()


def _host_forward(dims, x, residual, W, pinned=True, out=None):
    T, H = dims[:2]
    ws = moe.new_workspace(dims)
    x_dev = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    out_dev = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16)
        out = out.pin_memory() if pinned else out
    moe.moe_forward_host_io(dims, x, W, residual, out, x_dev, out_dev, ws)
    torch.cuda.synchronize()
    assert moe.moe_last_device_error(ws) == 0
    return out


@pytest.mark.parametrize("dims", CASES, ids=lambda d: "x".join(map(str, d)))
def test_host_io_parity(dims):
    x, residual, w, W = _layer(dims, 71 + dims[0])
    out = _host_forward(dims, x.pin_memory(), residual.pin_memory(), W)
    assert_close(out.float().numpy(), oracle.forward(dims, x, w, residual)["out"], f"moe_forward_host_io {dims}")
    assert torch.equal(out, _device_forward(dims, x, residual, W))


@pytest.mark.parametrize("dims", CASES, ids=lambda d: "x".join(map(str, d)))
def test_host_io_pageable_and_in_place(dims):
    x, residual, w, W = _layer(dims, 5 + dims[0])
    ref = _device_forward(dims, x, None, W)
    assert torch.equal(_host_forward(dims, x.clone(), None, W, pinned=False), ref)
    hx = x.clone().pin_memory()
    out = _host_forward(dims, hx, None, W, out=hx)  # the output replaces the host x
    assert out.data_ptr() == hx.data_ptr() and torch.equal(hx, ref)
    ref_r = _device_forward(dims, x, residual, W)
    hr = residual.clone()
    assert torch.equal(_host_forward(dims, x, hr, W, out=hr), ref_r)  # over the host residual


def test_host_io_refuses_device_buffers_as_host_rows():
    dims = CASES[1]
    x, residual, w, W = _layer(dims, 9)
    T, H = dims[:2]
    ws = moe.new_workspace(dims)
    x_dev = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    out_dev = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    host_out = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    with pytest.raises(ValueError, match="CPU tensors"):
        moe.moe_forward_host_io(dims, x.cuda(), W, None, host_out, x_dev, out_dev, ws)
    # through the C ABI: device memory as a host buffer, or host memory as device staging, is
    # refused before any copy
    lib = binding.load_library()
    d, cw = binding.Dims(*dims), W.to_c()
    hx = x.pin_memory()
    call = lambda hx_, hout, xd, od: lib.moe_forward_host_io(  # noqa: E731
        ctypes.byref(d), hx_, ctypes.byref(cw), None, hout, xd, od, ws.data_ptr(), ws.numel(), None)
    assert call(x_dev.data_ptr(), host_out.data_ptr(), x_dev.data_ptr(), out_dev.data_ptr()) == 1
    assert call(hx.data_ptr(), out_dev.data_ptr(), x_dev.data_ptr(), out_dev.data_ptr()) == 1
    assert call(hx.data_ptr(), host_out.data_ptr(), x_dev.data_ptr(), host_out.data_ptr()) == 1
    assert call(hx.data_ptr(), host_out.data_ptr(), hx.data_ptr(), out_dev.data_ptr()) == 1
    torch.cuda.synchronize()


def test_prepared_call_matches_the_entry():
    dims = CASES[0]
    x, residual, w, W = _layer(dims, 17)
    T, H = dims[:2]
    ws = moe.new_workspace(dims)
    x_dev = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    out_dev = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    call = moe.ForwardHostIO(dims, W, x_dev, out_dev, ws)
    hx, hr = x.pin_memory(), residual.pin_memory()
    outs = []
    for r in (None, hr, None):  # the same prepared call, with and without a residual
        out = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
        call(hx, out, r)
        torch.cuda.synchronize()
        outs.append(out)
    assert moe.moe_last_device_error(ws) == 0
    assert torch.equal(outs[0], _device_forward(dims, x, None, W))
    assert torch.equal(outs[1], _device_forward(dims, x, residual, W))
    assert torch.equal(outs[2], outs[0])
    with pytest.raises(ValueError, match="the layer needs"):
        call(hx[:, :8].contiguous(), outs[0])
