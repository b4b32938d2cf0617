"""In-kernel timeline of the one-token layer kernel.

    python -m sparse_moe_ffn_router_gb300.timeline [--layers 8] [--calls 64] [--replays 3]

Builds the MOE_TIMELINE variant of the library (libmoe_gb300_timeline.so; the kernel records
the global timer at ten fixed points of each CTA's call), runs `calls` one-token layer calls
over `layers` distinct seeded layers of the 2048 / 256-expert / top-8 / 512 shape in one CUDA
graph, and prints, for the last call of each replay, every event's minimum / median / maximum
over the CTAs in microseconds after the call's first CTA start. Needs a GPU; the stamps cost a
few hundred nanoseconds per call, so the per-layer time printed is a little above the
uninstrumented one.
"""
from __future__ import annotations

import argparse
import ctypes

import numpy as np

EVENTS = [
    "CTA start",
    "producer 0: weight-only items issued",
    "producer 0: previous kernel complete",
    "consumers: token row in registers",
    "a router score published",
    "warp 0: every CTA's router scores seen",
    "warp 0: routing known, producer released",
    "producer 0: every item issued",
    "consumers: every item done (combine starts)",
    "combine done",
]


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--calls", type=int, default=64)
    ap.add_argument("--replays", type=int, default=3)
    args = ap.parse_args(argv)

    import torch

    from . import binding
    from . import build as nbuild
    from . import synth
    from .workloads import WORKLOADS

    nbuild.LIB = nbuild.build(timeline=True)
    lib = binding.load_library(build_if_missing=False)
    lib.moe_timeline_read.restype = ctypes.c_int
    lib.moe_timeline_read.argtypes = [ctypes.c_void_p]
    ctas, nev = ctypes.c_int(), ctypes.c_int()
    lib.moe_timeline_shape(ctypes.byref(ctas), ctypes.byref(nev))

    wl = WORKLOADS["decode_T1"]
    dims = wl.dims
    dev = torch.device("cuda")
    layers = []
    for layer in range(args.layers):
        w = synth.make_weights(wl.H, wl.E, wl.I, wl.Is, wl.seed, layer, None, device=dev)
        layers.append((binding.Weights.from_dict(w), synth.make_x(wl.T, wl.H, wl.seed, layer, device=dev)))
    ws = binding.new_workspace(dims, dev)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)

    def step(i):
        W, x = layers[i % len(layers)]
        binding.moe_forward(dims, x, W, None, out, ws)

    for i in range(2 * args.layers):
        step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(args.calls):
            step(i)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(10):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    print(f"one-token layer, {args.calls} calls per graph: {a.elapsed_time(b) * 1e3 / (10 * args.calls):.2f} us per "
          f"call (timeline build)")
    print(f"device error word: {binding.moe_last_device_error(ws)}")
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    for r in range(args.replays):
        g.replay()
        torch.cuda.synchronize()
        tl = np.zeros(ctas.value * nev.value, np.uint64)
        if lib.moe_timeline_read(tl.ctypes.data) != 0:
            raise RuntimeError("moe_timeline_read failed")
        tl = tl.reshape(ctas.value, nev.value)[: min(nsm, ctas.value)].astype(np.int64)
        t0 = tl[:, 0].min()
        print(f"--- replay {r}: the last call, us after its first CTA start (min / median / max over CTAs)")
        for e, name in enumerate(EVENTS):
            v = tl[:, e]
            v = (v[(v >= t0) & (v - t0 < 10 ** 6)] - t0) / 1e3
            if len(v):
                print(f"{e:2d} {name:44s} {v.min():7.2f} {np.median(v):7.2f} {v.max():7.2f}   n={len(v)}")
        # the same CTA's time from one event to the next
        ok = ((tl >= t0) & (tl - t0 < 10 ** 6)).all(axis=1)
        d = np.diff(tl[ok], axis=1) / 1e3
        print(f"    per-CTA time from event e-1 to e (min / median / max over {int(ok.sum())} CTAs)")
        for e in range(1, len(EVENTS)):
            print(f"{e:2d} {'':44s} {d[:, e - 1].min():7.2f} {np.median(d[:, e - 1]):7.2f} {d[:, e - 1].max():7.2f}")


if __name__ == "__main__":
    main()
