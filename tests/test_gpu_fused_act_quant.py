"""The quantised GEMM1s with the gated activation and its dynamic
quantisation in the epilogue (grouped_gemm_w13 with fuse_act: FP8 128x128
block scales with fp32 or UE8M0 activation scales, MXFP4 W4A8, MXFP8) against
the two-step form of the same stage (GEMM1 to a bf16 h1,
then act_mul_quant): both round the sums to bf16, apply the activation in fp32
and quantise with the same scale rule, so codes and scales must agree bit for
bit on every row below num_post_padded.  Ragged expert loads, both
weight-scale forms (K % 512 == 0 stages them by TMA), one and several column
blocks, expert biases and the alpha / beta / clamp recipe."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import MoEConfig, make_inputs

from .gpu_util import np32

pytestmark = pytest.mark.gpu

RECIPE = (1.702, 1.0, 7.0)


def _ragged(quant, counts, H, I, seed, fmt="ue8m0"):
    E = len(counts)
    ids = np.concatenate([np.full(c, e, dtype=np.int32) for e, c in enumerate(counts)])
    np.random.default_rng(seed).shuffle(ids)
    M = len(ids)
    cfg = MoEConfig("fa", M=M, H=H, I=I, E=E, topk=1, quant=quant, routing="uniform", seed=seed,
                    act_scale_fmt=fmt)
    d = make_inputs(cfg, "cuda")
    d["topk_ids"] = torch.from_numpy(ids).view(M, 1).cuda()
    return cfg, d


@pytest.mark.parametrize("quant,fmt", [("fp8", "fp32"), ("fp8", "ue8m0"), ("mxfp4", "ue8m0"),
                                      ("mxfp8", "ue8m0")])
@pytest.mark.parametrize("counts,H,I,bias,recipe", [
    ([0, 1, 127, 128, 129, 300], 512, 256, False, None),    # staged weight scales
    ([0, 1, 127, 128, 129, 300], 640, 384, False, None),    # per-lane weight scales
    ([7, 0, 260], 1024, 128, True, None),                   # one column block, biases
    ([3, 200, 50, 0, 129], 512, 512, True, RECIPE),         # biases + gated recipe
])
def test_fused_act_matches_two_step(quant, fmt, counts, H, I, bias, recipe):
    cfg, d = _ragged(quant, counts, H, I, 31, fmt)
    p = moe.Problem.from_config(cfg, act_recipe=recipe)
    b = moe.stage_buffers(p)
    b13 = None
    if bias:
        g = torch.Generator().manual_seed(5)
        b13 = (torch.randn(cfg.E, 2 * I, generator=g) * 0.5).to(torch.bfloat16).cuda()
    moe.moe_align_permute(p, d["x"], d["topk_ids"], None, b["sorted_ids"], b["block_expert_ids"],
                          b["expert_offsets"], b["num_post_padded"], b["inv_perm"], b["x_perm"],
                          b["x_perm_scale"], b["align_ws"])
    # two steps: bf16 h1, then the activation kernel
    moe.grouped_gemm_w13_ex(p, b["x_perm"], b["x_perm_scale"], d["w13"], d["w13_scale"], b13,
                            b["block_expert_ids"], b["num_post_padded"], b["h1"])
    moe.act_mul_quant(p, b["h1"], b["num_post_padded"], b["z"], b["z_scale"])
    # fused, into buffers pre-filled so that an unwritten element shows up
    zf = torch.full_like(b["z"], 0x7F)
    zsf = torch.full_like(b["z_scale"], float("nan"))
    moe.grouped_gemm_w13_ex(p, b["x_perm"], b["x_perm_scale"], d["w13"], d["w13_scale"], b13,
                            b["block_expert_ids"], b["num_post_padded"], zf, zsf, fuse_act=True)
    assert moe.moe_sync_status() == 0
    n = int(b["num_post_padded"].item())
    assert n > 0
    assert np.array_equal(np32(zf)[:n], np32(b["z"])[:n])
    assert np.array_equal(np32(zsf)[:n], np32(b["z_scale"])[:n])


def test_fused_act_requires_scale_output():
    cfg, d = _ragged("mxfp4", [5, 9], 256, 128, 3)
    p = moe.Problem.from_config(cfg)
    b = moe.stage_buffers(p)
    with pytest.raises(moe.MoEError):
        moe.grouped_gemm_w13(p, b["x_perm"], b["x_perm_scale"], d["w13"], d["w13_scale"],
                             b["block_expert_ids"], b["num_post_padded"], b["z"], None,
                             fuse_act=True)
