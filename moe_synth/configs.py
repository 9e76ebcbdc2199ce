"""The five workloads the library is checked and measured on.

Shapes: Mixtral-8x7B-class experts (H=4096, I=14336, E=8, top-2) at prefill and
decode token counts, a DeepSeek-class FP8 layer (H=7168, I=2048, E=256, top-8)
with skewed routing, the same DeepSeek-class shape with MXFP4 weights, and
with MXFP8 (1x32) weights and activations.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class MoEConfig:
    name: str
    M: int            # tokens
    H: int            # hidden size (K of GEMM1, N of GEMM2)
    I: int            # expert intermediate size (GEMM1 N = 2I)
    E: int            # experts
    topk: int
    quant: str        # "bf16" | "fp8" | "mxfp4" | "mxfp8"
    routing: str      # "softmax" | "skew" | "uniform"
    seed: int
    block_size: int = 128
    act_scale_fmt: str = "fp32"   # "fp32" | "ue8m0" (activation scales of quantised modes)
    apply_router_weight_on_input: bool = False
    invalid_frac: float = 0.0     # fraction of (token, slot) ids replaced by -1

    @property
    def R(self) -> int:
        return self.M * self.topk

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


CONFIGS = {
    "tiny": MoEConfig("tiny", M=16, H=256, I=128, E=8, topk=2, quant="bf16",
                      routing="softmax", seed=1),
    "mixtral": MoEConfig("mixtral", M=4096, H=4096, I=14336, E=8, topk=2,
                         quant="bf16", routing="softmax", seed=2),
    "decode": MoEConfig("decode", M=64, H=4096, I=14336, E=8, topk=2,
                        quant="bf16", routing="softmax", seed=3),
    "dsfp8": MoEConfig("dsfp8", M=8192, H=7168, I=2048, E=256, topk=8,
                       quant="fp8", routing="skew", seed=4),
    "mxfp4": MoEConfig("mxfp4", M=2048, H=7168, I=2048, E=256, topk=8,
                       quant="mxfp4", routing="uniform", seed=5,
                       act_scale_fmt="ue8m0"),
    "mxfp8": MoEConfig("mxfp8", M=8192, H=7168, I=2048, E=256, topk=8, quant="mxfp8",
                       routing="skew", seed=6, act_scale_fmt="ue8m0"),
}


def get_config(name: str) -> MoEConfig:
    return CONFIGS[name]
