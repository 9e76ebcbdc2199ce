"""Failure detection of the GEMM kernels without faulting the GPU.

Every mbarrier wait in the GEMMs is bounded by wall clock.  The debug hook
moe_debug_set_watchdog(limit_ns, never_arrive=True) makes the TMA producer
leave its first pipeline stage unarmed, so the MMA thread's wait runs out
after limit_ns.  The kernel must then record MOE_ERR_DEVICE_TIMEOUT in the
device error word, drain what it issued, free its tensor memory and return;
the host reads the status with moe_sync_status, and the same CUDA context
must keep working (a normal call right after gives correct results)."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import MoEConfig, make_inputs
from oracle import experts

from .gpu_util import (BF16_TOL, QUANT_TOL, bf16_gemm_form, check_close, flip_allowance, np32,
                       oracle_inputs)

pytestmark = pytest.mark.gpu

CASES = {
    "bf16": MoEConfig("wd16", M=200, H=512, I=256, E=4, topk=2, quant="bf16", routing="softmax",
                      seed=81),
    "fp8": MoEConfig("wd8", M=200, H=512, I=256, E=4, topk=2, quant="fp8", routing="softmax",
                     seed=82),
    # prepacked weight scales: the block-scaled GEMM's pair form needs them
    "mxfp8": MoEConfig("wdm8", M=200, H=512, I=256, E=4, topk=2, quant="mxfp8",
                       routing="softmax", seed=83, act_scale_fmt="ue8m0"),
    # W4A8: a warp of its own copies the scale operands into tensor memory
    "mxfp4": MoEConfig("wdm4", M=200, H=512, I=256, E=4, topk=2, quant="mxfp4",
                       routing="softmax", seed=84, act_scale_fmt="ue8m0"),
}


def _fused(cfg, d):
    if cfg.quant in ("mxfp4", "mxfp8"):
        p = moe.Problem.from_config(cfg, weight_scales_prepacked=True)
        if "w13_scale_packed" not in d:
            q = moe.Problem.from_config(cfg)
            d["w13_scale_packed"] = torch.empty(moe.moe_prepacked_scale_bytes(q, 0),
                                                dtype=torch.uint8, device="cuda")
            d["w2_scale_packed"] = torch.empty(moe.moe_prepacked_scale_bytes(q, 1),
                                               dtype=torch.uint8, device="cuda")
            moe.moe_prepack_weights(q, d["w13_scale"], d["w2_scale"], d["w13_scale_packed"],
                                    d["w2_scale_packed"])
        ws = torch.empty(moe.moe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
        y = torch.empty_like(d["x"])
        moe.fused_experts(p, d["x"], d["w13"], d["w13_scale_packed"], d["w2"],
                          d["w2_scale_packed"], d["topk_weights"], d["topk_ids"], y, ws)
        return y
    p = moe.Problem.from_config(cfg)
    ws = torch.empty(moe.moe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(d["x"])
    moe.fused_experts(p, d["x"], d["w13"], d["w13_scale"], d["w2"], d["w2_scale"],
                      d["topk_weights"], d["topk_ids"], y, ws)
    return y


@pytest.mark.parametrize("name,form", [("bf16", "single"), ("bf16", "pairs"), ("fp8", "auto"),
                                       ("fp8", "pairs"), ("mxfp8", "auto"), ("mxfp8", "pairs"),
                                       ("mxfp4", "auto"), ("mxfp4", "pairs")])
def test_wait_that_runs_out_reports_timeout_and_context_survives(name, form):
    with bf16_gemm_form(form):
        _timeout_then_recover(name)


def _timeout_then_recover(name):
    cfg = CASES[name]
    d = make_inputs(cfg, "cuda")
    assert moe.moe_sync_status() == 0
    try:
        moe.moe_debug_set_watchdog(50_000_000, never_arrive=True)   # 50 ms
        _fused(cfg, d)
        assert moe.moe_sync_status() == 4          # MOE_ERR_DEVICE_TIMEOUT
    finally:
        moe.moe_debug_set_watchdog(0, never_arrive=False)
    assert moe.moe_sync_status() == 0              # the error word was cleared
    # the context still works: a normal call gives the oracle's answer
    y = _fused(cfg, d)
    assert moe.moe_sync_status() == 0
    ref, items, w = experts.fused_experts_per_token(
        **oracle_inputs(d), quant=cfg.quant, act_scale_fmt=cfg.act_scale_fmt, return_items=True)
    check_close(np32(y), ref, BF16_TOL if cfg.quant == "bf16" else QUANT_TOL, f"{name} watchdog",
                flip_allowance(ref, items, w))
