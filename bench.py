#!/usr/bin/env python3
"""Benchmark of the GB300 sparse MoE feed-forward layer.

`python bench.py --gpus N --steps K --warmup W` times K steps of the layer on synthetic,
seeded inputs and prints ONE JSON line (rank 0). A step is one full pass of the layer
(router scores, softmax/top-K/renorm, dispatch, gate_up+SwiGLU, down+scale, fixed-order
combine) over one batch of tokens, called through the C ABI (`moe_forward`).

Headline workload: decode of one token at the full layer shape (H=2048, 256 experts, top-8,
inner 512). Steps cycle through 8 distinct seeded layers (12.9 GB of weights), so the ~58 MB
of weights a step touches were last read 8 steps earlier (>= 460 MB ago) and are not served
from the 129 MB L2. Weights and inputs are resident in HBM before timing starts.

Extra keys: `roofline` (dominant kernel: algorithmic bytes per launch over its CUDA-event
duration inside the timed region, against the measured HBM copy bandwidth), `e2e` (the same
metric through moe_forward_host_io: x read from pinned host memory and the output written
back to it by the library, inside the timed region), `cpu_baseline` (the fp64 C oracle on the host cores on a bounded sample of the same
workload), `clocks` (nvidia-smi samples taken during the timed region), `layer` (the whole
layer's fractions of the HBM and tensor peaks and of its binding roofline), `also` (the
decode T=64, prefill T=4096 and 40-layer stack workloads, shorter runs of the same
measurement, each with the load-balancing statistics call and the bf16-score variant timed
beside it), `host_experts` (decode with the routed experts in pinned host memory, fetched
over the host link per step).

`--impl reference` times the oracle (the only reference implementation: the pages publish
no code) on the host cores for the same workload and metric.

With N > 1 (torchrun), every rank runs the same per-GPU workload on its own GPU (tokens are
independent; no collective on the data path): value = tokens of all ranks / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from sparse_moe_ffn_router_gb300 import synth  # noqa: E402
from sparse_moe_ffn_router_gb300.workloads import RMSNORM_EPS, WORKLOADS  # noqa: E402

METRIC = "MoE-layer tokens/s"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "decode_T1"
ROTATE = 8
KERNEL_NAMES = ["router_scores", "router_topk", "dispatch_local", "dispatch_scan", "dispatch_scatter", "gate_up",
                "down", "combine", "rmsnorm", "shared_gate", "gather", "gemm_plan", "decode_fused", "fetch_experts",
                "copy_rows"]
HOST_LAYERS = 4  # layers cycled through with host-resident experts (their touched experts exceed L2)


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=0,
                   help="steps per timed repeat (default 512); the repeat runs until --min-seconds of timed work")
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    p.add_argument("--min-seconds", type=float, default=1.0, help="timed work of the headline workload, in seconds")
    p.add_argument("--also-seconds", type=float, default=0.5, help="timed work of each extra workload, in seconds")
    p.add_argument("--also", default="decode_T8,decode_T64,prefill_T4096_zipf,stack40_decode_T32",
                   help="comma-separated extra workloads reported under 'also' ('none' to skip)")
    p.add_argument("--cpu-budget", type=float, default=10.0,
                   help="seconds of oracle work for cpu_baseline (0: no oracle baseline, e.g. for profiling runs)")
    p.add_argument("--no-graph", action="store_true", help="time plain calls instead of CUDA-graph replays")
    p.add_argument("--rotate", type=int, default=ROTATE,
                   help="distinct layers cycled through by small-T workloads (keeps weights out of L2)")
    a = p.parse_args()
    a.warmup = max(a.warmup, 3)
    return a


# ---------------------------------------------------------------------------------------
# distributed plumbing (one process per GPU)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def max_over_ranks(v: float) -> float:
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())
    return v


# ---------------------------------------------------------------------------------------
# peaks, clocks


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (read + write) of `kernel` on `workload` from profiles/
    ncu_traffic.json, or None when absent or recorded for another version of the kernel's
    source file (each record names the file and its SHA-1)."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f).get(kernel, {}).get(workload)
        if not rec:
            return None
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            sha = hashlib.sha1(f.read()).hexdigest()
    except (OSError, KeyError, ValueError, AttributeError, TypeError):
        return None
    if rec.get("source_sha1") != sha:
        return None
    return rec.get("dram_bytes_per_launch")


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi samples (every 200 ms) of this process's GPU during a region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            sel = str(device_index)
        self.sel = sel

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.sel, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def mark(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def __exit__(self, *exc):
        time.sleep(0.25)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        from datetime import datetime
        rows = []
        try:
            for line in open(self.path):
                f = [c.strip() for c in line.split(",")]
                if len(f) >= 10 and f[2].replace(".", "").isdigit():
                    try:
                        ts = datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    except ValueError:
                        ts = None
                    rows.append((ts, f[1:]))
        except OSError:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        t0, t1 = getattr(self, "t0", None), getattr(self, "t1", None)
        inside = [r for ts, r in rows if ts is not None and t0 is not None and t1 is not None and t0 <= ts <= t1]
        use = inside or [r for _, r in rows]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        sm = [float(r[1]) for r in use]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in use for n, v in zip(names, r[5:9]) if v.lower().startswith("active")})
        pw = [float(r[3]) for r in use if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(use[0][2]), "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": len(inside), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------------------
# the workloads on the GPU


class LayerSet:
    """n distinct seeded layers of a workload, resident on the GPU, with their inputs."""

    def __init__(self, wl, n_layers: int, device):
        import sparse_moe_ffn_router_gb300 as moe
        self.moe = moe
        self.wl = wl
        self.dims = wl.dims
        self.device = device
        self.layers = []
        for l in range(n_layers):
            w = synth.make_weights(wl.H, wl.E, wl.I, wl.Is, wl.seed, l, wl.zipf_s, device=device)
            x = synth.make_x(wl.T, wl.H, wl.seed, l, device=device)
            self.layers.append((moe.Weights.from_dict(w), x))
        self.ws = moe.new_workspace(self.dims, device)
        self.out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=device)
        self._groups = None

    def step(self, layer: int):
        W, x = self.layers[layer % len(self.layers)]
        self.moe.moe_forward(self.dims, x, W, None, self.out, self.ws)

    def routed_groups(self) -> list[list[int]]:
        """Per layer: rows of each touched expert (for the algorithmic byte count)."""
        if self._groups is None:
            self._groups = [route_counts(self.moe, self.dims, x, W, self.device) for W, x in self.layers]
        return self._groups


def route_counts(moe, dims, x, W, device) -> list[int]:
    """Rows routed to each touched expert for one call (moe_route on its own workspace)."""
    T, H, E, K = dims[:4]
    ws = moe.new_workspace(dims, device)
    ids = torch.empty(T, K, dtype=torch.int32, device=device)
    tw = torch.empty(T, K, dtype=torch.float32, device=device)
    counts = torch.empty(E, dtype=torch.int32, device=device)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=device)
    perm = torch.empty(T * K, dtype=torch.int32, device=device)
    moe.moe_route(dims, x, W, ids, tw, counts, offsets, perm, ws)
    return [int(c) for c in counts.cpu().tolist() if c > 0]


def algorithmic(dims, groups: list[int]) -> dict:
    """Bytes each kernel must move at least (the method's bytes), and the layer's flops, for
    one call; `impl_*` adds what this implementation stages on top.

    Method bytes: gate_up reads each touched expert's [2I, H] block and the shared [2Is, H]
    once, x once, and writes h; down reads each touched [H, I] block and the shared [H, Is]
    once and reads h; the layer adds the router [E+1, H], x and out. Implementation bytes:
    down writes Y (bf16 from 256 tokens, fp32 below) for the fixed-order combine, which reads
    it back (the gate_up GEMM gathers its token rows from x, which stays in L2 across the K
    experts that read a row)."""
    T, H, E, K, I, Is = dims[:6]
    P = T * K
    n = len(groups)
    ysz = 2 if T >= 256 else 4
    h_bytes = 2 * (P * I + T * Is)
    gate_up = 2 * (n * 2 * I * H + 2 * Is * H) + 2 * T * H + h_bytes
    down = 2 * (n * H * I + H * Is) + h_bytes
    router = 2 * (E + 1) * H + 2 * T * H
    layer_bytes = 2 * ((E + 1) * H + n * 3 * I * H + 3 * Is * H) + 2 * 2 * T * H
    flops = 2 * T * (E + 1) * H + 2 * P * 3 * I * H + 2 * T * 3 * Is * H
    impl_gate_up = gate_up
    impl_down = down + ysz * (P + T) * H
    combine = ysz * (P + T) * H + 2 * T * H
    return dict(gate_up=gate_up, down=down, router_scores=router, decode_fused=layer_bytes, layer=layer_bytes,
                flops=flops, impl_gate_up=impl_gate_up, impl_down=impl_down, impl_combine=combine,
                impl_decode_fused=layer_bytes)


def trace_kernels(moe, names, n):
    ev = {k: ([torch.cuda.Event(enable_timing=True) for _ in range(n)],
              [torch.cuda.Event(enable_timing=True) for _ in range(n)]) for k in names}
    # torch creates the CUDA event on its first record; each start/stop pair is recorded back
    # to back, so a kernel that never launches reads ~0 ms
    for a, b in ev.values():
        for x, y in zip(a, b):
            x.record()
            y.record()
    torch.cuda.synchronize()
    for k, (a, b) in ev.items():
        moe.moe_set_trace(k, a, b)
    return ev


def clear_traces(moe):
    for k in KERNEL_NAMES:
        moe.moe_set_trace(k)


def kernel_ms(ev, n) -> dict:
    return {k: sum(a[i].elapsed_time(b[i]) for i in range(n)) / n for k, (a, b) in ev.items()}


def graph_plan(steps: int, n_layers: int, gmax: int) -> tuple[int, list[int]]:
    """A CUDA graph of G steps (G divides the requested step count, G <= gmax) and the layer
    each of its steps runs. Consecutive steps never run the same layer, also across the
    boundary between two replays (then the last step takes the next layer instead)."""
    G = max(d for d in range(1, min(steps, gmax) + 1) if steps % d == 0)
    layers = [i % n_layers for i in range(G)]
    if n_layers > 2 and G > 1 and layers[-1] == layers[0]:
        layers[-1] = (layers[-1] + 1) % n_layers
    return G, layers


def percentile(v: list[float], q: float) -> float:
    s = sorted(v)
    if len(s) == 1:
        return s[0]
    x = q * (len(s) - 1)
    i = int(math.floor(x))
    j = min(i + 1, len(s) - 1)
    return s[i] + (s[j] - s[i]) * (x - i)


def timed_regions(run_region, min_total_s: float, min_repeats: int, sampler=None) -> list[float]:
    """Repeat one timed region (exactly the requested steps) until about min_total_s of timed
    work, each repeat between CUDA events on the launching stream, with a barrier and a
    synchronize on both sides of the whole timed span; milliseconds of each repeat (max over
    ranks)."""
    # one untimed region sizes the repeat count
    t0 = time.perf_counter()
    run_region()
    torch.cuda.synchronize()
    one = max(time.perf_counter() - t0, 1e-6)
    reps = int(min(100000, max(min_repeats, math.ceil(min_total_s / one))))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(True)
    ev[0].record()
    for r in range(reps):
        run_region()
        ev[r + 1].record()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(False)
    barrier()
    return [max_over_ranks(ev[r].elapsed_time(ev[r + 1])) for r in range(reps)]


def spread(ms_regions: list[float], steps: int) -> dict:
    per = [m / steps for m in ms_regions]
    return {"repeats": len(per), "median_ms_per_step": round(statistics.median(per), 6),
            "p10_ms_per_step": round(percentile(per, 0.1), 6), "p90_ms_per_step": round(percentile(per, 0.9), 6),
            "timed_s_total": round(sum(ms_regions) / 1e3, 3)}


def time_layer_set(ls: LayerSet, steps: int, warmup: int, peaks: dict, clocks_index=None, min_total_s: float = 1.0,
                   graph: bool = True, gmax: int = 4096, auto_steps: int = 512):
    """Warm-up (all kernels traced, to find the dominant one), then the timed region: exactly
    `steps` steps (a CUDA graph of G steps, G dividing `steps`, replayed steps/G times; plain
    calls without graph), repeated until about min_total_s of timed work. Reported: the
    median repeat (tokens/s, ms per step) with p10/p90 over the repeats. The dominant
    kernel's duration: for one launch per step, the timed repeats over their launches; else
    per-launch CUDA events from a second graph of the same steps, replayed once after the
    timed region (no event node inside the timed graph). Returns a result dict."""
    moe = ls.moe
    nl = len(ls.layers)
    ev = trace_kernels(moe, KERNEL_NAMES, warmup)
    for i in range(warmup):
        ls.step(i)
    torch.cuda.synchronize()
    warm = kernel_ms(ev, warmup)
    clear_traces(moe)
    dominant = max(warm, key=warm.get)
    if steps <= 0:
        steps = auto_steps
    G, order = graph_plan(steps, nl, gmax) if graph else (steps, [i % nl for i in range(steps)])
    if graph:
        g = torch.cuda.CUDAGraph()
        n0 = moe.moe_launch_count()
        with torch.cuda.graph(g):
            for l in order:
                ls.step(l)
        per_graph = moe.moe_launch_count() - n0
        g.replay()
        torch.cuda.synchronize()
        run = lambda: [g.replay() for _ in range(steps // G)]  # noqa: E731
        launches_per_region = per_graph * (steps // G)
    else:
        n0 = moe.moe_launch_count()
        for l in order:
            ls.step(l)
        torch.cuda.synchronize()
        launches_per_region = moe.moe_launch_count() - n0
        run = lambda: [ls.step(l) for l in order]  # noqa: E731
    sampler = ClockSampler(clocks_index) if clocks_index is not None else None
    if sampler:
        sampler.__enter__()
    regions = timed_regions(run, min_total_s, 5, sampler)
    if sampler:
        sampler.__exit__(None, None, None)
    sp = spread(regions, steps)
    ms = sp["median_ms_per_step"] * steps  # the median repeat
    one_launch = launches_per_region == steps
    if one_launch:
        dom_ms = ms / steps
        dom_src = "median timed repeat / launches"
    else:
        ev = trace_kernels(moe, [dominant], G)
        if graph:
            g_trace = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_trace):
                for l in order:
                    ls.step(l)
            clear_traces(moe)
            g_trace.replay()
            torch.cuda.synchronize()
        else:
            for l in order[:G]:
                ls.step(l)
            torch.cuda.synchronize()
        dom_ms = kernel_ms(ev, G)[dominant]
        dom_src = "per-launch events"
        clear_traces(moe)
    groups = ls.routed_groups()
    per_step = [algorithmic(ls.dims, groups[l % nl]) for l in order]
    alg_bytes = sum(p.get(dominant, 0) for p in per_step) / len(order)
    impl_bytes = sum(p.get("impl_" + dominant, 0) for p in per_step) / len(order)
    layer_bytes = sum(p["layer"] for p in per_step) / len(order)
    flops = per_step[0]["flops"]
    T = ls.dims[0]
    # the device error word of the workspace (0: no non-finite score, no timed-out wait)
    dev_err = moe.moe_last_device_error(ls.ws)
    res = dict(steps=steps, ms_per_step=ms / steps, tokens_per_s=T * steps / (ms / 1e3),
               launches=launches_per_region * sp["repeats"], launches_per_step=launches_per_region / steps,
               spread=sp, device_error=dev_err, graph_steps=G if graph else None,
               dominant=dominant, dominant_ms=dom_ms, dominant_ms_source=dom_src, warm_kernel_ms=warm, graph=graph,
               unique_experts=sum(len(groups[l % nl]) for l in order) / len(order),
               layer_bytes=layer_bytes, layer_flops=flops)
    if alg_bytes:
        ach = alg_bytes / (dom_ms * 1e-3) / 1e9
        res["roofline"] = {"bound": "hbm", "kernel": dominant, "achieved": round(ach, 1),
                           "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
                           "traffic": None, "bytes_per_launch": int(alg_bytes),
                           "impl_bytes_per_launch": int(impl_bytes),
                           "duration_us": round(dom_ms * 1e3, 3), "duration_source": dom_src,
                           "peak_source": peaks["source"]}
    layer_gbs = layer_bytes / (ms / steps * 1e-3) / 1e9
    res["layer_hbm_frac"] = round(layer_gbs / peaks["hbm_gbs"], 4)
    res["layer_tensor_frac"] = round(flops / (ms / steps * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)
    # the layer against its binding roofline: max(bytes / HBM peak, flops / tensor peak) / time
    res["layer_binding_frac"] = max(res["layer_hbm_frac"], res["layer_tensor_frac"])
    if sampler:
        res["clocks"] = sampler.summary()
    return res


def time_stats(ls: LayerSet, peaks: dict, n: int = 20, reps: int = 10) -> dict:
    """moe_router_stats (load-balancing statistics) on one layer: a CUDA graph of n calls,
    replayed reps times. Bytes: router weights and x read, the score matrix written and read
    back, the ids read."""
    moe = ls.moe
    T, H, E, K = ls.dims[:4]
    dev = ls.out.device
    P = torch.empty(E, dtype=torch.float32, device=dev)
    f = torch.empty(E, dtype=torch.float32, device=dev)
    loss = torch.empty(4, dtype=torch.float32, device=dev)
    W, x = ls.layers[0]
    for _ in range(3):
        moe.moe_router_stats(ls.dims, x, W, P, f, loss, ls.ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(n):
            moe.moe_router_stats(ls.dims, x, W, P, f, loss, ls.ws)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / (n * reps)
    nbytes = 2 * (E + 1) * H + 2 * T * H + 2 * 4 * T * (E + 1) + 4 * T * K
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us_per_call": round(us, 2), "tokens_per_s": round(T / (us * 1e-6), 1),
            "device_error": moe.moe_last_device_error(ls.ws),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "bytes_per_call": nbytes}}


def time_variant(ls: LayerSet, flags: int, n: int = 32, reps: int = 5) -> dict:
    """moe_forward with the dims flags (MOE_FLAG_BF16_SCORES: bf16-typed router and shared-gate
    scores) and without them, over the same rotating layers: n steps, a CUDA graph replayed
    reps times up to 64 tokens, plain launches above."""
    moe = ls.moe
    T = ls.dims[0]

    def run(dims) -> float:
        def step(i):
            W, x = ls.layers[i % len(ls.layers)]
            moe.moe_forward(dims, x, W, None, ls.out, ls.ws)

        for i in range(3):
            step(i)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if T <= 64:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(n):
                    step(i)
            g.replay()
            torch.cuda.synchronize()
            a.record()
            for _ in range(reps):
                g.replay()
            b.record()
        else:
            a.record()
            for i in range(n * reps):
                step(i)
            b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (n * reps)

    base = run(tuple(ls.dims))
    var = run(tuple(ls.dims) + (flags,))
    return {"ms_per_step": round(var, 5), "tokens_per_s": round(T / (var * 1e-3), 1),
            "default_ms_per_step": round(base, 5), "device_error": moe.moe_last_device_error(ls.ws)}


def time_host_experts(wl, device, n: int = 32, reps: int = 5) -> dict:
    """moe_forward_host_experts: the routed experts (gate_up, down) of HOST_LAYERS layers in
    pinned host memory, router and shared expert in HBM, one device shadow for all layers.
    Step time over the rotating layers (a CUDA graph of n steps replayed reps times), and the
    fetch kernel's share: the touched experts' bytes over its event-timed duration (the host
    link's achieved rate)."""
    import sparse_moe_ffn_router_gb300 as moe
    T, H, E, K, I, Is = wl.dims
    layers, nbytes = [], []
    for l in range(HOST_LAYERS):
        w = synth.make_weights(H, E, I, Is, wl.seed, l, wl.zipf_s)
        x = synth.make_x(T, H, wl.seed, l, device=device)
        dev = {k: (None if v is None else v.to(device)) for k, v in w.items()}
        dev["gate_up"], dev["down"] = w["gate_up"].pin_memory(), w["down"].pin_memory()
        layers.append((moe.Weights.from_dict(dev), x))
    ws = moe.new_workspace(wl.dims, device)
    shadow = torch.zeros(moe.moe_expert_shadow_size(wl.dims), dtype=torch.uint8, device=device)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=device)
    # experts each layer touches (the bytes its fetch copies)
    for W, x in layers:
        ids = torch.empty(T, K, dtype=torch.int32, device=device)
        tw = torch.empty(T, K, dtype=torch.float32, device=device)
        counts = torch.empty(E, dtype=torch.int32, device=device)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=device)
        perm = torch.empty(T * K, dtype=torch.int32, device=device)
        Wd = moe.Weights(W.router_w, W.router_b, W.shared_gate_up, W.shared_gate_up, W.shared_gate_up, W.shared_down,
                         W.shared_gate)  # routing reads the router and the shared gate only
        moe.moe_route(wl.dims, x, Wd, ids, tw, counts, offsets, perm, ws)
        nbytes.append(int((counts > 0).sum().item()) * (2 * I * H + H * I) * 2)

    def step(i):
        W, x = layers[i % HOST_LAYERS]
        moe.moe_forward_host_experts(wl.dims, x, W, None, out, shadow, ws)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            step(i)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (n * reps)
    ev = trace_kernels(moe, ["fetch_experts"], n)
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        for i in range(n):
            step(i)
    g2.replay()
    torch.cuda.synchronize()
    clear_traces(moe)
    fetch_ms = kernel_ms(ev, n)["fetch_experts"]
    fetched = sum(nbytes[i % HOST_LAYERS] for i in range(n)) / n
    err = moe.moe_last_device_error(ws)
    del layers, shadow
    link = fetched / (fetch_ms * 1e-3) / 1e9
    ce = copy_engine_h2d_gbs(device)
    return {"tokens_per_s": round(T / (ms * 1e-3), 1), "ms_per_step": round(ms, 5),
            "expert_bytes_per_step": int(fetched), "fetch_ms": round(fetch_ms, 5),
            "host_link_gbs": round(link, 1), "copy_engine_h2d_gbs": round(ce, 1),
            "fetch_frac_of_copy_engine": round(link / ce, 3), "layers": HOST_LAYERS, "device_error": err}


def copy_engine_h2d_gbs(device, nbytes: int = 512 << 20, reps: int = 3) -> float:
    """The host link's rate as the copy engine sees it on this machine: one pinned-host to device
    copy of 512 MB (cudaMemcpyAsync through torch), best of `reps`. The fetch kernel's rate is
    reported beside it as a fraction."""
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=device)
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    best = 0.0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(reps):
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (a.elapsed_time(b) * 1e6))
    del src, dst
    return best


def time_e2e(ls: LayerSet, steps: int, warmup: int) -> dict:
    """Same metric through the public call with host buffers (moe_forward_host_io, prepared
    once per layer as a ForwardHostIO): per step, the library brings x in from pinned host
    memory, runs the layer, and puts the output back in pinned host memory (at T = 1 the
    one-token kernel reads and writes the host rows itself; otherwise copies to and from
    device staging around the layer). Also reports the host time to issue one step, taken over the first steps of the
    timed loop while the launch queue is still short (a host time close to the step time
    means the loop is issue-bound)."""
    moe = ls.moe
    T, H = ls.dims[:2]
    hx = [x.cpu().pin_memory() for _, x in ls.layers]
    hout = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    xd = torch.empty(T, H, dtype=torch.bfloat16, device=ls.device)
    calls = [moe.ForwardHostIO(ls.dims, W, xd, ls.out, ls.ws) for W, _ in ls.layers]

    def step(i):
        calls[i % len(calls)](hx[i % len(hx)], hout)

    for i in range(warmup):
        step(i)
    barrier()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    n_host = min(steps, 64)
    t0 = time.perf_counter()
    for i in range(n_host):
        step(warmup + i)
    t1 = time.perf_counter()
    for i in range(n_host, steps):
        step(warmup + i)
    stop.record()
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(start.elapsed_time(stop))
    return dict(value=T * steps / (ms / 1e3), ms_per_step=ms / steps, h2d=T * H * 2, d2h=T * H * 2,
                host_us_per_step=(t1 - t0) / n_host * 1e6)


class StackSet:
    """The 40-layer stack: x_{l+1} = x_l + MoE_l(RMSNorm(x_l)), one distinct layer each. The
    residual stream ping-pongs between two buffers (layer l reads one and writes the other),
    so a step is only the layers' own launches."""

    def __init__(self, wl, device):
        import sparse_moe_ffn_router_gb300 as moe
        self.moe = moe
        self.wl = wl
        self.dims = wl.dims
        self.device = device
        self.layers = [moe.Weights.from_dict(synth.make_weights(wl.H, wl.E, wl.I, wl.Is, wl.seed, l, None,
                                                                device=device)) for l in range(wl.layers)]
        self.x0 = synth.make_x(wl.T, wl.H, wl.seed, 0, device=device, tag="x_stack")
        self.buf = [torch.empty_like(self.x0), torch.empty_like(self.x0)]
        self.xn = torch.empty_like(self.x0)
        self.ws = moe.new_workspace(self.dims, device)
        self._groups = None

    def step(self, i: int = 0, groups: list | None = None):
        x = self.x0
        for l, W in enumerate(self.layers):
            out = self.buf[l % 2]
            self.moe.moe_rmsnorm(self.dims, x, None, RMSNORM_EPS, self.xn)
            if groups is not None:
                groups.append(route_counts(self.moe, self.dims, self.xn, W, self.device))
            self.moe.moe_forward(self.dims, self.xn, W, x, out, self.ws)
            x = out

    def routed_groups(self) -> list[list[int]]:
        """Per layer: rows of each touched expert of one step (all steps route alike)."""
        if self._groups is None:
            g = []
            self.step(0, g)
            torch.cuda.synchronize()
            self._groups = g
        return self._groups


def time_stack(ss: StackSet, steps: int, warmup: int, peaks: dict, min_total_s: float = 0.5) -> dict:
    """The stack's step as one CUDA graph (40 x (RMSNorm + layer)), replayed `steps` times per
    timed repeat; bytes per step: every layer's router, touched experts, shared expert, its
    input, residual and output rows, and the RMSNorm's read and write."""
    moe = ss.moe
    for i in range(warmup):
        ss.step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    n0 = moe.moe_launch_count()
    with torch.cuda.graph(g):
        ss.step(0)
    per_step = moe.moe_launch_count() - n0
    g.replay()
    torch.cuda.synchronize()
    regions = timed_regions(lambda: [g.replay() for _ in range(steps)], min_total_s, 3)
    sp = spread(regions, steps)
    ms = sp["median_ms_per_step"]
    T, H = ss.dims[:2]
    groups = ss.routed_groups()
    nbytes = sum(algorithmic(ss.dims, gr)["layer"] + 2 * T * H + 4 * T * H for gr in groups)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return dict(ms_per_step=ms, tokens_per_s=T / (ms * 1e-3), layers=len(ss.layers), steps=steps, spread=sp,
                launches_per_step=per_step, device_error=moe.moe_last_device_error(ss.ws),
                unique_experts_per_layer=round(sum(len(gr) for gr in groups) / len(groups), 2),
                roofline={"bound": "hbm", "kernel": "whole step (40 layers)", "achieved": round(gbs, 1),
                          "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                          "bytes_per_step": int(nbytes), "peak_source": peaks["source"]})


# ---------------------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and --impl reference)


def oracle_steps(wl, steps: int, warmup: int, budget_s=None, device=None, tokens=None) -> dict:
    """Time the fp64 C oracle (OpenMP over tokens on the host's threads) on steps of the
    workload with its layer-0 weights: each step is the whole layer for the first `tokens`
    tokens of the workload's x (all T by default). For the layer stack one layer stands for
    each of its layers (all cost the same), so a step takes layers x one layer's time."""
    import oracle
    dev = device if device is not None else "cpu"
    w = synth.make_weights(wl.H, wl.E, wl.I, wl.Is, wl.seed, 0, wl.zipf_s, device=dev)
    hw = {k: (None if v is None else v.cpu()) for k, v in w.items()}
    del w
    T = wl.T if tokens is None else max(1, min(tokens, wl.T))
    x = synth.make_x(wl.T, wl.H, wl.seed, 0)[:T].contiguous()
    dims = (T,) + tuple(wl.dims[1:])
    for _ in range(warmup):
        oracle.forward(dims, x, hw)
    if budget_s is not None:
        t0 = time.perf_counter()
        oracle.forward(dims, x, hw)
        one = time.perf_counter() - t0
        steps = max(1, min(steps, int(budget_s / max(one, 1e-6))))
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.forward(dims, x, hw)
    dt = time.perf_counter() - t0
    cores = min(T, oracle.num_threads())
    return dict(value=T * steps / (dt * wl.layers), steps=steps, seconds=dt, cores=cores, tokens=T,
                host_cores=os.cpu_count())


def cpu_baseline(wl, budget_s: float, device, tokens=None) -> dict:
    r = oracle_steps(wl, 10 ** 6, 1, budget_s=budget_s, device=device, tokens=tokens)
    what = f"{r['steps']} oracle steps of {r['tokens']} of the workload's {wl.T} token(s), layer-0 weights"
    if wl.layers > 1:
        what += f", one layer standing for each of the {wl.layers}"
    return {"value": round(r["value"], 3), "unit": UNIT, "cores": r["cores"], "host_cores": r["host_cores"],
            "kind": "oracle", "sample": f"{what}; {r['seconds']:.1f} s of fp64 C oracle work"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    r = oracle_steps(wl, args.steps if args.steps > 0 else 100, args.warmup, device=dev)
    sample = f"{r['steps']} steps of {wl.name} ({wl.T} token(s) each), layer-0 weights, fp64 C oracle"
    line = {"impl": "reference", "metric": METRIC, "value": round(r["value"], 3), "unit": UNIT, "n_gpus": world,
            "steps": r["steps"], "warmup": args.warmup, "ms_per_step": round(r["seconds"] / r["steps"] * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded SplitMix64 + Box-Muller, bf16)",
            "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "E": wl.E, "K": wl.K, "I": wl.I, "Is": wl.Is},
            "cpu_baseline": {"value": round(r["value"], 3), "unit": UNIT, "cores": r["cores"],
                             "host_cores": r["host_cores"], "kind": "oracle", "sample": sample},
            "e2e": {"value": round(r["value"], 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------


def also_entry(r: dict, world: int) -> dict:
    return {"tokens_per_s": round(r["tokens_per_s"] * world, 2), "ms_per_step": round(r["ms_per_step"], 5),
            "steps": r["steps"], "timing": r["spread"], "device_error": r["device_error"],
            "roofline": r.get("roofline"), "hbm_frac_of_layer_bytes": r["layer_hbm_frac"],
            "tensor_frac": r["layer_tensor_frac"], "binding_frac": r["layer_binding_frac"],
            "unique_experts_per_step": r["unique_experts"], "launches_per_step": r["launches_per_step"],
            "kernel_ms_warmup": {k: round(v, 5) for k, v in r["warm_kernel_ms"].items()}}


def main():
    args = parse_args()
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the layer has no CPU path)")
    import sparse_moe_ffn_router_gb300 as moe
    moe.load_library()
    device = torch.device("cuda", torch.cuda.current_device())
    peaks = load_peaks()
    wl = WORKLOADS[args.workload]
    if wl.layers > 1:
        raise SystemExit("use the stack workload under --also")
    n_rot = max(1, args.rotate) if wl.T <= 32 else 1
    ls = LayerSet(wl, n_rot, device)
    main_res = time_layer_set(ls, args.steps, args.warmup, peaks, clocks_index=torch.cuda.current_device(),
                              graph=not args.no_graph, min_total_s=args.min_seconds)
    if main_res.get("roofline"):
        main_res["roofline"]["traffic"] = ncu_traffic(main_res["roofline"]["kernel"], wl.name)
    e2e_steps = int(min(50000, max(main_res["steps"], 0.5 / (main_res["ms_per_step"] * 1e-3))))
    e2e = time_e2e(ls, e2e_steps, args.warmup)
    value = main_res["tokens_per_s"] * world
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": main_res["steps"],
        "warmup": args.warmup, "ms_per_step": round(main_res["ms_per_step"], 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64 + Box-Muller, bf16; random-init weights of the full layer shape)",
        "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "E": wl.E, "K": wl.K, "I": wl.I, "Is": wl.Is,
                   "layers_rotated": n_rot,
                   "l2": ("inputs larger than L2: steps cycle through %d distinct layers (%.1f GB)"
                          % (n_rot, n_rot * wl.weight_bytes_per_layer() / 1e9)) if n_rot > 1 else
                   "inputs larger than L2 (%.2f GB of weights touched per step)" % (main_res["layer_bytes"] / 1e9),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "cuda_graph": main_res["graph"]},
        "timing": dict(main_res["spread"], graph_steps=main_res["graph_steps"],
                       note="value and ms_per_step: the median of the timed repeats, each exactly `steps` steps"),
        "roofline": main_res.get("roofline"),
        "e2e": {"value": round(e2e["value"] * world, 3), "unit": UNIT, "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": round(e2e["ms_per_step"], 6), "steps": e2e_steps,
                "host_us_per_step": round(e2e["host_us_per_step"], 2)},
        "gpu_launches": main_res["launches"],
        "device_error": main_res["device_error"],
        "clocks": main_res.get("clocks"),
        "layer": {"unique_experts_per_step": main_res["unique_experts"],
                  "hbm_frac_of_layer_bytes": main_res["layer_hbm_frac"],
                  "tensor_frac": main_res["layer_tensor_frac"],
                  "binding_frac": main_res["layer_binding_frac"],
                  "launches_per_step": main_res["launches_per_step"],
                  "kernel_ms_warmup": {k: round(v, 5) for k, v in main_res["warm_kernel_ms"].items()}},
    }
    del ls
    torch.cuda.empty_cache()
    also = {}
    names = [] if args.also in ("", "none") else [n for n in args.also.split(",") if n]
    cpu_also = rank == 0 and world == 1 and args.cpu_budget > 0
    for name in names:
        w2 = WORKLOADS[name]
        if w2.layers > 1:
            ss = StackSet(w2, device)
            r = time_stack(ss, 3, 2, peaks, min_total_s=args.also_seconds)
            also[name] = {"tokens_per_s": round(r["tokens_per_s"] * world, 2), "ms_per_step": round(r["ms_per_step"], 4),
                          "steps": r["steps"], "timing": r["spread"], "layers": r["layers"],
                          "launches_per_step": r["launches_per_step"], "device_error": r["device_error"],
                          "unique_experts_per_layer": r["unique_experts_per_layer"], "roofline": r["roofline"],
                          "cuda_graph": True}
            del ss
        else:
            ls2 = LayerSet(w2, ROTATE if w2.T <= 32 else 1, device)
            r = time_layer_set(ls2, 0, 3, peaks, graph=not args.no_graph, min_total_s=args.also_seconds,
                               auto_steps=64 if w2.T >= 256 else 512)
            if r.get("roofline"):
                r["roofline"]["traffic"] = ncu_traffic(r["roofline"]["kernel"], w2.name)
            also[name] = also_entry(r, world)
            if name != "decode_T8":
                also[name]["router_stats"] = time_stats(ls2, peaks)
                also[name]["bf16_scores"] = time_variant(ls2, ls2.moe.FLAG_BF16_SCORES)
            del ls2
        torch.cuda.empty_cache()
        if cpu_also:
            also[name]["cpu_baseline"] = cpu_baseline(w2, args.cpu_budget / 2, device,
                                                      tokens=256 if w2.T > 256 else None)
    line["also"] = also
    # routed experts resident in host memory, fetched over the host link per step
    # (with the extra workloads only: the short runs behind the ncu launch lists skip it)
    host = {}
    for name in ("decode_T1", "decode_T64"):
        if names and (name == wl.name or name in names):
            host[name] = time_host_experts(WORKLOADS[name], device)
            torch.cuda.empty_cache()
    line["host_experts"] = host
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_budget, device, tokens=256 if wl.T > 256 else None)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
