"""Seeded synthetic inputs for the fused MoE expert forward.

This module only draws inputs: hidden states, router outputs (top-k ids and
weights) and expert weights in the storage formats the path consumes.  It holds
none of the expert computation, so both the CPU oracle and the CUDA library can
be fed from it without sharing any arithmetic of the method.

Workload shapes follow the page "fused_moe.py 分析" (FlagDoc), §1.1-1.2 (the
router produces top-k weights/ids, experts are gated MLPs with w13 [E, 2I, H]
and w2 [E, H, I]) and the page "Blackwell 上的 DeepGEMM FusedMoE（vLLM）", TL;DR
table (FP8 128x128 block weights; MXFP4 E2M1 weights with E8M0 scales per 32).
"""
from .configs import CONFIGS, MoEConfig, get_config  # noqa: F401
from .gen import make_inputs, make_routing  # noqa: F401
