"""Expert parallelism (sparse_moe_ffn_router_gb300/ep.py) in two, three and four gloo processes
on CPU.

Rank r of N owns experts [floor(r*E/N), floor((r+1)*E/N)) and is home to tokens
[floor(r*T/N), floor((r+1)*T/N)) of a seeded layer (three ranks split both unevenly). Each rank routes its own tokens with the oracle, runs the exchange (counts, dispatch,
expert outputs back, fixed-order combine) with the expert math restated in fp64 numpy, and
the tests check, against the oracle's routing and layer output for all T tokens at once:
  - routing, bit for bit: the (expert, token, slot) triples each owner receives are exactly
    the oracle's pairs whose expert it owns, in (expert, token, slot) order per source rank,
    and each received row is the token's row, bit for bit;
  - the output of every token within 1e-9 (relative to the output's scale) of oracle.forward.
One case routes evenly; one biases the router so that one rank receives no rows at all.
Unmeasured on hardware: the same calls would run over NCCL on GPUs."""
from __future__ import annotations

import os
import pickle
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

DIMS = (16, 64, 8, 2, 32, 32)  # T (all ranks), H, E, K, I, Is


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer(bias_low: bool, world: int):
    from sparse_moe_ffn_router_gb300 import synth
    T, H, E, K, I, Is = DIMS
    w = synth.make_weights(H, E, I, Is, seed=77)
    if bias_low:
        # experts of rank 0 never win: every pair goes to the other ranks
        b = torch.zeros(E, dtype=torch.float32)
        b[: E // world] = -30.0
        w["router_b"] = b.to(torch.bfloat16)
    x = synth.make_x(T, H, seed=78)
    return w, x


def _swiglu(rows: np.ndarray, gate_up: np.ndarray, down: np.ndarray) -> np.ndarray:
    I = down.shape[1]
    g = rows @ gate_up[:I].T
    u = rows @ gate_up[I:].T
    return (g / (1.0 + np.exp(-g)) * u) @ down.T


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.float().double().numpy()


def _rank_main(rank: int, world: int, port: int, bias_low: bool, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    from sparse_moe_ffn_router_gb300 import ep

    dist.init_process_group("gloo", rank=rank, world_size=world)
    T, H, E, K, I, Is = DIMS
    t0, t1 = rank * T // world, (rank + 1) * T // world
    w, x = _layer(bias_low, world)
    xr = x[t0:t1]
    dims_r = (t1 - t0,) + DIMS[1:]
    r = oracle.route(dims_r, xr, w["router_w"], w["router_b"])
    taps = oracle.forward(dims_r, xr, w, taps=True)  # the shared gate and shared output of the home tokens
    gu, dn = _f64(w["gate_up"]), _f64(w["down"])
    res = ep.ep_layer(xr, torch.from_numpy(r["ids"]), torch.from_numpy(r["w"]), torch.from_numpy(taps["sg"]),
                      torch.from_numpy(taps["ys"]),
                      lambda e, rows: torch.from_numpy(_swiglu(_f64(rows), gu[e], dn[e])), E)
    res["rows"] = res["rows"].view(torch.int16)  # bf16 bit patterns (numpy has no bf16)
    with open(os.path.join(out_dir, f"rank{rank}.pkl"), "wb") as f:
        pickle.dump({k: (v.numpy() if torch.is_tensor(v) else v) for k, v in res.items()}, f)
    dist.destroy_process_group()


def _run(tmp_path, bias_low: bool, world: int = 2):
    import oracle
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, bias_low, str(tmp_path)), nprocs=world, start_method="spawn",
                       join=True)
    got = [pickle.load(open(tmp_path / f"rank{r}.pkl", "rb")) for r in range(world)]
    w, x = _layer(bias_low, world)
    T, H, E, K, I, Is = DIMS
    home = [(r * T // world, (r + 1) * T // world) for r in range(world)]
    ref_route = oracle.route(DIMS, x, w["router_w"], w["router_b"])
    ref = oracle.forward(DIMS, x, w)["out"]
    xb = x.view(torch.int16).numpy()
    for owner in range(world):
        g = got[owner]
        lo, hi = owner * E // world, (owner + 1) * E // world
        # what the owner must receive from each source rank, in (expert, token, slot) order
        want = []
        for src in range(world):
            s0, s1 = home[src]
            pairs = [(int(ref_route["ids"][t, k]), t - s0, k) for t in range(s0, s1)
                     for k in range(K) if lo <= ref_route["ids"][t, k] < hi]
            want += [(src,) + p for p in sorted(pairs)]
        have = [(int(s),) + tuple(int(v) for v in m) for s, m in zip(g["src"], g["meta"])]
        assert have == want, f"owner {owner}: received pairs"
        for (src, e, tl, k), row in zip(have, g["rows"]):
            assert np.array_equal(row, xb[home[src][0] + tl]), f"owner {owner}: row of token {home[src][0] + tl}"
        assert int(g["recv_counts"].sum()) == len(want)
    out = np.concatenate([got[r]["out"] for r in range(world)])
    scale = np.abs(ref).max()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-9 * scale)
    return got


@pytest.mark.parametrize("world", [2, 3, 4])
def test_expert_parallel_exchange_matches_the_oracle(tmp_path, world):
    got = _run(tmp_path, bias_low=False, world=world)
    assert all(int(g["recv_counts"].sum()) > 0 for g in got)


def test_expert_parallel_exchange_with_an_idle_owner(tmp_path):
    got = _run(tmp_path, bias_low=True)
    assert int(got[0]["recv_counts"].sum()) == 0  # rank 0's experts receive nothing
    assert int(got[1]["recv_counts"].sum()) == DIMS[0] * DIMS[3]


def test_dispatch_order_is_the_stable_expert_sort():
    from sparse_moe_ffn_router_gb300 import ep
    ids = torch.tensor([[3, 1], [1, 0], [2, 3]])
    order, counts = ep.dispatch_order(ids, 4, 2)
    # pairs p = t*K + k: expert 0 <- p3; expert 1 <- p1, p2; expert 2 <- p4; expert 3 <- p0, p5
    assert order.tolist() == [3, 1, 2, 4, 0, 5]
    assert counts.tolist() == [3, 3]
    # 6 experts over 4 ranks: [0, 1), [1, 3), [3, 4), [4, 6)
    assert ep.owners(torch.arange(6), 6, 4).tolist() == [0, 1, 1, 2, 3, 3]
    order, counts = ep.dispatch_order(ids, 6, 4)
    assert order.tolist() == [3, 1, 2, 4, 0, 5] and counts.tolist() == [1, 3, 2, 0]
    with pytest.raises(ValueError):
        ep.owners(torch.arange(2), 2, 3)  # more ranks than experts
