"""Layer calls back to back on one stream, with no synchronisation between them, as a model runs
its layers: each call's token rows are the previous call's output, and all calls share one
workspace. Consecutive calls' kernels overlap (programmatic dependent launch: a call's set-up
and weight-only copies run while the previous call finishes; each kernel waits for the
previous one before it reads its output or the workspace). After one synchronisation every
call's output is compared with the oracle run on that call's own input (the previous call's
output, read back from the GPU), so an input read too early or workspace state overwritten
too soon shows up as a wrong layer. Layers cycle through distinct seeded weights."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import sparse_moe_ffn_router_gb300 as moe
from sparse_moe_ffn_router_gb300 import synth
from sparse_moe_ffn_router_gb300.workloads import WORKLOADS
from tests.gpu_helpers import assert_close
from tests.inputs import gap_controlled_x

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,calls,n_weights,sample", [
    ("decode_T1", 12, 4, None),
    ("decode_T8", 8, 4, None),
    ("prefill_T4096_zipf", 3, 2, 128),
])
def test_chained_calls_back_to_back(name, calls, n_weights, sample):
    wl = WORKLOADS[name]
    dims = wl.dims
    T, H = wl.T, wl.H
    dev = torch.device("cuda")
    weights = [synth.make_weights(H, wl.E, wl.I, wl.Is, wl.seed, l, wl.zipf_s, device=dev) for l in range(n_weights)]
    Ws = [moe.Weights.from_dict(w) for w in weights]
    x0, _ = gap_controlled_x(dims, weights[0]["router_w"].cpu(),
                             None if weights[0]["router_b"] is None else weights[0]["router_b"].cpu(), wl.seed, 0)
    ws = moe.new_workspace(dims, dev)
    xs = [x0.to(dev)] + [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(calls)]
    for c in range(calls):  # call c reads xs[c] and writes xs[c + 1]
        moe.moe_forward(dims, xs[c], Ws[c % n_weights], None, xs[c + 1], ws)
    torch.cuda.synchronize()
    assert moe.moe_last_device_error(ws) == 0
    host = [{k: (None if v is None else v.cpu()) for k, v in w.items()} for w in weights]
    rows = np.arange(T) if sample is None else np.random.default_rng(7).choice(T, sample, replace=False)
    rows.sort()
    sub = (len(rows),) + tuple(dims[1:])
    for c in range(calls):
        x_in = xs[c].cpu()[rows]
        ref = oracle.forward(sub, x_in, host[c % n_weights])["out"]
        got = xs[c + 1].cpu()[rows].float().numpy()
        assert_close(got, ref, f"{name}: call {c} of {calls}")


def test_chained_host_row_calls_back_to_back():
    """One-token calls with the token rows in pinned host memory (moe_forward_host_io), back to
    back with no synchronisation: call c reads host row c, which call c - 1's kernel wrote over
    the host link, and a residual row written by the call before that."""
    wl = WORKLOADS["decode_T1"]
    dims = wl.dims
    T, H = wl.T, wl.H
    calls, n_weights = 10, 3
    dev = torch.device("cuda")
    weights = [synth.make_weights(H, wl.E, wl.I, wl.Is, wl.seed, l, wl.zipf_s, device=dev) for l in range(n_weights)]
    Ws = [moe.Weights.from_dict(w) for w in weights]
    x0, _ = gap_controlled_x(dims, weights[0]["router_w"].cpu(),
                             None if weights[0]["router_b"] is None else weights[0]["router_b"].cpu(), wl.seed, 0)
    ws = moe.new_workspace(dims, dev)
    xd = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    od = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    hs = [x0.clone().pin_memory()] + [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(calls)]
    for c in range(calls):  # call c reads hs[c] (and hs[c - 1] as its residual) and writes hs[c + 1]
        moe.moe_forward_host_io(dims, hs[c], Ws[c % n_weights], hs[c - 1] if c else None, hs[c + 1], xd, od, ws)
    torch.cuda.synchronize()
    assert moe.moe_last_device_error(ws) == 0
    host = [{k: (None if v is None else v.cpu()) for k, v in w.items()} for w in weights]
    for c in range(calls):
        ref = oracle.forward(dims, hs[c].clone(), host[c % n_weights], hs[c - 1].clone() if c else None)["out"]
        assert_close(hs[c + 1].float().numpy(), ref, f"host rows: call {c} of {calls}")
