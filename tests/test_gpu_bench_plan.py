"""The launches bench.py times per step (its stage plan, through the staged
entry points) give exactly the output of fused_experts: same kernels, same
order, so y agrees bit for bit.  Small shapes of every mode, a decode-sized
bf16 case (GEMM2 in K slices) and an SM-pair-sized one."""
import pytest
import torch

import bench
import mixture_experts_ffn_align_gb300 as moe
from moe_synth import MoEConfig, make_inputs

pytestmark = pytest.mark.gpu

CASES = {
    "bf16_sliced": MoEConfig("pb", M=64, H=512, I=1024, E=8, topk=2, quant="bf16",
                             routing="softmax", seed=91),
    "bf16_pairs": MoEConfig("pp", M=2048, H=256, I=256, E=4, topk=2, quant="bf16",
                            routing="softmax", seed=92),
    "fp8": MoEConfig("pf", M=96, H=512, I=256, E=8, topk=4, quant="fp8", routing="softmax",
                     seed=93),
    "mxfp4": MoEConfig("pm", M=96, H=512, I=256, E=8, topk=4, quant="mxfp4",
                       routing="uniform", seed=94, act_scale_fmt="ue8m0"),
    "mxfp8": MoEConfig("p8", M=96, H=512, I=256, E=8, topk=4, quant="mxfp8",
                       routing="uniform", seed=95, act_scale_fmt="ue8m0"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_bench_plan_matches_fused_experts(name):
    cfg = CASES[name]
    d = make_inputs(cfg, "cuda")
    p = moe.Problem.from_config(cfg)
    b = moe.stage_buffers(p)
    stream = torch.cuda.current_stream()
    plan = bench._stage_plan(moe, p, cfg, d, b, stream)
    for _, fn in plan:
        fn()
    ws = torch.empty(moe.moe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(d["x"])
    moe.fused_experts(p, d["x"], d["w13"], d["w13_scale"], d["w2"], d["w2_scale"],
                      d["topk_weights"], d["topk_ids"], y, ws)
    assert moe.moe_sync_status() == 0
    names = [n for n, _ in plan]
    if name == "bf16_sliced":
        assert "gemm2_split_k" in names and moe.moe_gemm2_splits(p) > 1
    assert torch.equal(b["y"], y), names
