"""The synthetic MoE workloads (shapes, formats, routing rules, seeds).

Each is a stand-in for a model the Pulsar / Strata pages run, at that
model's MoE-layer shape; weights and inputs are random (see synth/__init__.py).
"""
from __future__ import annotations

from dataclasses import dataclass

from .layout import FMT_Q4K, FMT_Q2K

ROUTE_SOFTMAX = 0
ROUTE_SIGMOID = 1


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    I: int
    E: int
    k: int
    S: int             # shared experts
    route: int
    fmt: int
    layers: int
    T: int             # tokens per layer per step
    seed: int
    bias_std: float = 0.0   # per-expert router logit bias (skewed popularity) when > 0

    def desc(self, T_max=None):
        return dict(H=self.H, I=self.I, E=self.E, top_k=self.k, n_shared=self.S, route=self.route,
                    fmt=self.fmt, T_max=T_max or self.T)

    def with_T(self, T):
        return Workload(**{**self.__dict__, "T": T, "name": f"{self.name.rsplit('_t', 1)[0]}_t{T}"})


WORKLOADS = {
    # tiny single layer, the oracle finishes in seconds
    "tiny_h512_e16k2_i256_t4": Workload("tiny_h512_e16k2_i256_t4", 512, 256, 16, 2, 0, ROUTE_SOFTMAX, FMT_Q4K,
                                        1, 4, 0),
    # Qwen3.6-35B-A3B-shaped decode: 40 layers, top-8 of 256 softmax + 1 shared, Q4_K-style, batch 1
    "decode_h2048_e256k8s1_i512_q4k_l40_t1": Workload("decode_h2048_e256k8s1_i512_q4k_l40_t1", 2048, 512, 256, 8, 1,
                                                      ROUTE_SOFTMAX, FMT_Q4K, 40, 1, 1),
    # Strata-like MTP verify window: 48 layers, top-10 of 512 sigmoid + 1 shared, Q2_K-style, 4 tokens
    "verify_h4096_e512k10s1_i1024_q2k_l48_t4": Workload("verify_h4096_e512k10s1_i1024_q2k_l48_t4", 4096, 1024, 512,
                                                        10, 1, ROUTE_SIGMOID, FMT_Q2K, 48, 4, 2),
    # Hy3-295B-like wide experts: one layer, top-8 of 192 softmax with a skewed router, T in 1..16
    "wide_h6144_e192k8_i2048_q4k_t16": Workload("wide_h6144_e192k8_i2048_q4k_t16", 6144, 2048, 192, 8, 0,
                                                ROUTE_SOFTMAX, FMT_Q4K, 1, 16, 3, bias_std=2.0),
    # long-prompt prefill chunk through one layer: 8192 tokens, top-10 of 512 sigmoid + 1 shared
    "prefill_h4096_e512k10s1_i1024_q4k_t8192": Workload("prefill_h4096_e512k10s1_i1024_q4k_t8192", 4096, 1024, 512,
                                                        10, 1, ROUTE_SIGMOID, FMT_Q4K, 1, 8192, 4),
}

DEFAULT_BENCH = "decode_h2048_e256k8s1_i512_q4k_l40_t1"
