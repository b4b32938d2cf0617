"""The bounded device waits give up, report MOE_ERR_TIMEOUT, and leave the library usable.

A testing aid of the C ABI (moe_test_set_wait) shortens the time limit of the waits to 2 ms
and holds one signal back, so that one wait of each kind runs out:
  - the one-token kernel's poll of the router scores that the other CTAs publish as tagged
    words (CTA 1 never publishes its scores);
  - the streaming gate_up kernel's wait on a ring stage's mbarrier (CTA 0 never loads its
    first stage).
Nothing faults or hangs: the call ends within the shortened limits, the workspace's error word
reads MOE_ERR_TIMEOUT, and after moe_workspace_init the next call matches the oracle again."""
from __future__ import annotations

import time

import pytest
import torch

import oracle
import sparse_moe_ffn_router_gb300 as moe
from tests.gpu_helpers import Layer, assert_close, run_forward

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000
MOE_ERR_TIMEOUT = 6


@pytest.mark.parametrize("T,suppress", [(1, moe.TEST_SUPPRESS_SCORE), (16, moe.TEST_SUPPRESS_STAGE)],
                         ids=["score-poll", "ring-mbarrier"])
def test_wait_runs_out_and_the_layer_recovers(T, suppress):
    dims = (T, 2048, 256, 8, 512, 512)
    L = Layer(dims, seed=500 + T)
    ws = moe.new_workspace(dims)
    out = torch.empty(T, dims[1], dtype=torch.bfloat16, device="cuda")
    run_forward(dims, L.xd, L.W, ws=ws, out=out)  # kernels loaded, the call path warm
    assert moe.moe_last_device_error(ws) == 0
    try:
        moe.moe_test_set_wait(LIMIT_NS, suppress)
        t0 = time.perf_counter()
        moe.moe_forward(dims, L.xd, L.W, None, out, ws)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        moe.moe_test_set_wait()  # normal operation for every later call
    assert moe.moe_last_device_error(ws) == MOE_ERR_TIMEOUT
    assert elapsed < 0.5, f"the call took {elapsed:.3f} s: the 2 ms limit was not applied"
    moe.moe_workspace_init(ws)
    ref = oracle.forward(dims, L.x, L.host_weights())
    out2, _ = run_forward(dims, L.xd, L.W, ws=ws)
    assert moe.moe_last_device_error(ws) == 0
    assert_close(out2.float().cpu().numpy(), ref["out"], f"T={T} after the timeout and moe_workspace_init")
