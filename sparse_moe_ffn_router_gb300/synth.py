"""Seeded synthetic inputs for the MoE layer, shared by the CUDA path's tests and benchmark
and by the oracle's tests.

This module holds none of the layer's arithmetic: it only draws numbers. Every value comes
from a counter-based generator, so any element can be reproduced from (seed, layer, tensor
tag, attempt, flat index) alone:

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
  OOPSLA 2014): output i of a stream with key k is mix(k + (i + 1) * 0x9E3779B97F4A7C15),
  where mix is the published SplitMix64 finaliser.
* Box-Muller (1958): two uniforms u1 in (0, 1], u2 in [0, 1) taken from the top 24 and the
  next 24 bits of one 64-bit draw give n = sqrt(-2 ln u1) * cos(2 pi u2) ~ N(0, 1), computed
  in fp32, scaled by the tensor's standard deviation and rounded to bf16 (nearest-even).

The integer part is exact on every device; the fp32 transcendental step may differ in the
last bit between CPU and GPU, so a test always hands the oracle host copies of the very
tensors the kernels read.
"""
from __future__ import annotations

import math

import torch

_MASK64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_CHUNK = 1 << 25

# Tensor tags of the key derivation.
TAGS = {"x": 1, "router_w": 2, "router_b": 3, "gate_up": 4, "down": 5, "shared_gate_up": 6,
        "shared_down": 7, "shared_gate": 8, "zipf_rank": 9, "x_stack": 10,
        # streams of the exact-score test inputs (small-integer values, see tests/inputs.py)
        "x_exact": 11, "router_w_exact": 12, "shared_gate_exact": 13, "router_b_exact": 14}


def _signed(v: int) -> int:
    v &= _MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def mix64(z: int) -> int:
    """SplitMix64 finaliser on a Python int (reference form)."""
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def splitmix64_py(key: int, i: int) -> int:
    """Output i of the counter-based stream with key ``key`` (reference form)."""
    return mix64(key + (i + 1) * _GOLDEN)


def stream_key(seed: int, layer: int, tag: str, attempt: int = 0) -> int:
    """64-bit key of one tensor's stream."""
    k = mix64(seed * 0x632BE59BD9B4E019 + 0x1F123BB5)
    k = mix64(k ^ (layer * 0x8CB92BA72F3D8DD7 + 0x2545F491))
    k = mix64(k ^ (TAGS[tag] * 0xD1B54A32D192ED03 + 0x4F1BBCDC))
    return mix64(k ^ (attempt * 0xA0761D6478BD642F + 0x27D4EB2F))


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def splitmix64(idx: torch.Tensor, key: int) -> torch.Tensor:
    """Vectorised SplitMix64 over int64 counters ``idx`` (wrap-around int64 arithmetic)."""
    z = idx + 1
    z = z * _signed(_GOLDEN) + _signed(key)
    z = (z ^ _lsr(z, 30)) * _signed(_M1)
    z = (z ^ _lsr(z, 27)) * _signed(_M2)
    return z ^ _lsr(z, 31)


def _normals_from_bits(z: torch.Tensor) -> torch.Tensor:
    u1 = (_lsr(z, 40) + 1).to(torch.float32) * (2.0 ** -24)
    u2 = (_lsr(z, 16) & 0xFFFFFF).to(torch.float32) * (2.0 ** -24)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def normal_bf16(shape, std: float, key: int, device="cpu", start: int = 0) -> torch.Tensor:
    """bf16 tensor of N(0, std^2) values, element i (row-major) from counter start + i."""
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        idx = torch.arange(start + c0, start + c1, dtype=torch.int64, device=device)
        out[c0:c1] = (_normals_from_bits(splitmix64(idx, key)) * std).to(torch.bfloat16)
    return out.view(*shape)


def uniform_u64(n: int, key: int, device="cpu") -> torch.Tensor:
    """n raw 64-bit draws (int64 bit patterns)."""
    return splitmix64(torch.arange(n, dtype=torch.int64, device=device), key)


# ----------------------------------------------------------------------------------------
# Layer inputs


def make_x(T: int, H: int, seed: int, layer: int = 0, attempts=None, device="cpu", tag: str = "x") -> torch.Tensor:
    """Token activations x [T, H] ~ N(0, 1) in bf16.

    Row t uses the stream of ``attempts[t]`` (default 0) and counters t*H .. t*H+H-1, so a
    test can redraw single rows (for example to keep routing scores apart) without moving
    any other row."""
    x = normal_bf16((T, H), 1.0, stream_key(seed, layer, tag, 0), device)
    if attempts is not None:
        attempts = torch.as_tensor(attempts, dtype=torch.int64)
        for a in sorted(set(int(v) for v in attempts.tolist()) - {0}):
            rows = torch.nonzero(attempts == a).flatten().tolist()
            key = stream_key(seed, layer, tag, a)
            for t in rows:
                x[t] = normal_bf16((H,), 1.0, key, device, start=t * H)
    return x


def zipf_ranks(E: int, seed: int, layer: int = 0) -> torch.Tensor:
    """A seeded random permutation r of 1..E (r[e] = popularity rank of expert e)."""
    z = uniform_u64(E, stream_key(seed, layer, "zipf_rank"))
    order = torch.argsort(z)  # int64 bit patterns are distinct with overwhelming probability
    r = torch.empty(E, dtype=torch.int64)
    r[order] = torch.arange(1, E + 1, dtype=torch.int64)
    return r


# Scale of the Zipf router bias. With b_e = -ZIPF_ALPHA * s * ln(r_e), s = 1.1, the seeded
# prefill workload (T=4096, H=2048, E=256, K=8, router std 0.02) gives a fitted log-log slope
# of the sorted expert loads close to -s; the calibration is printed by the routing tests.
ZIPF_ALPHA = 0.42


def zipf_bias(E: int, s: float, seed: int, layer: int = 0, alpha: float = ZIPF_ALPHA) -> torch.Tensor:
    """Router bias b_e = -alpha * s * ln(r_e) (bf16) that skews expert load toward Zipf(s)."""
    r = zipf_ranks(E, seed, layer).to(torch.float64)
    return (-alpha * s * torch.log(r)).to(torch.bfloat16)


def make_weights(H: int, E: int, I: int, Is: int, seed: int, layer: int = 0, zipf_s=None,
                 device="cpu", router_std: float = 0.02) -> dict:
    """All weight tensors of one layer, bf16, [Out, In] row-major.

    Router W ~ N(0, router_std^2); every other weight ~ N(0, 1/fan_in) (std 1/sqrt(fan_in)),
    fan_in = H for gate_up, shared gate_up and the shared gate, fan_in = I (Is) for down."""
    k = lambda tag: stream_key(seed, layer, tag)  # noqa: E731
    w = {
        "router_w": normal_bf16((E, H), router_std, k("router_w"), device),
        "router_b": None,
        "gate_up": normal_bf16((E, 2 * I, H), 1.0 / math.sqrt(H), k("gate_up"), device),
        "down": normal_bf16((E, H, I), 1.0 / math.sqrt(I), k("down"), device),
        "shared_gate_up": normal_bf16((2 * Is, H), 1.0 / math.sqrt(H), k("shared_gate_up"), device),
        "shared_down": normal_bf16((H, Is), 1.0 / math.sqrt(Is), k("shared_down"), device),
        "shared_gate": normal_bf16((1, H), 1.0 / math.sqrt(H), k("shared_gate"), device),
    }
    if zipf_s is not None:
        w["router_b"] = zipf_bias(E, zipf_s, seed, layer).to(device)
    return w
