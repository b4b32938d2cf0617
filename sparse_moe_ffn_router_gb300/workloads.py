"""The synthetic workloads of the MoE layer: shapes, seeds and routing skew.

Full layer shape: H=2048, 256 experts, top-8, expert inner 512, shared inner 512
("Qwen3.6 35B-A3B", Generics: H, Experts, TopK, ExpertInner, SharedInner; merged gate_up
[256, 1024, 2048] in "Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256 Experts).
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    K: int
    I: int
    Is: int
    seed: int
    layers: int = 1
    zipf_s: float | None = None
    note: str = ""

    @property
    def dims(self):
        return (self.T, self.H, self.E, self.K, self.I, self.Is)

    def weight_bytes_per_layer(self) -> int:
        H, E, I, Is = self.H, self.E, self.I, self.Is
        return 2 * (E * H + E * 2 * I * H + E * H * I + 2 * Is * H + H * Is + H)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_T8", 8, 512, 32, 4, 128, 128, seed=0,
                 note="smallest instance: T=8, H=512, 32 experts, top-4, inner 128"),
        Workload("decode_T1", 1, 2048, 256, 8, 512, 512, seed=1, note="decode, one token, full layer shape"),
        Workload("decode_T8", 8, 2048, 256, 8, 512, 512, seed=5, note="decode batch of 8 tokens, full layer shape"),
        Workload("decode_T64", 64, 2048, 256, 8, 512, 512, seed=2,
                 note="decode batch of 64 tokens, near-uniform routing"),
        Workload("prefill_T4096_zipf", 4096, 2048, 256, 8, 512, 512, seed=3, zipf_s=1.1,
                 note="prefill of 4096 tokens, router bias skewing expert load toward Zipf(1.1)"),
        Workload("stack40_decode_T32", 32, 2048, 256, 8, 512, 512, seed=4, layers=40,
                 note="40 distinct full-shape layers chained by RMSNorm(eps 1e-6) + residual, 32 tokens"),
    ]
}

RMSNORM_EPS = 1e-6
