"""GPU parity of the epilogue variants (expert biases, the router weight in
GEMM2's epilogue with a summing reduce, the gated activation recipe) through
fused_experts_ex and the stage entry points, bf16 (both tile forms), FP8 and
MXFP4, against the oracle with the same options."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import MoEConfig, make_inputs
from oracle import codecs, experts

from .gpu_util import (BF16_TOL, QUANT_TOL, bf16_gemm_form, check_close, flip_allowance, np32,
                       oracle_inputs)

pytestmark = pytest.mark.gpu

RECIPE = (1.702, 1.0, 7.0)


def _biases(cfg, seed):
    g = torch.Generator().manual_seed(seed)
    b13 = (torch.randn(cfg.E, 2 * cfg.I, generator=g) * 0.5).to(torch.bfloat16).cuda()
    b2 = (torch.randn(cfg.E, cfg.H, generator=g) * 0.5).to(torch.bfloat16).cuda()
    return b13, b2


def _run(cfg, d, p, b13, b2):
    ws = torch.empty(moe.moe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(d["x"])
    moe.fused_experts_ex(p, d["x"], d["w13"], d["w13_scale"], b13, d["w2"], d["w2_scale"], b2,
                         d["topk_weights"], d["topk_ids"], y, ws)
    assert moe.moe_sync_status() == 0
    return y


def _oracle(cfg, d, b13, b2, in_gemm2, recipe, tokens=None):
    y, items, w = experts.fused_experts_per_token(
        **oracle_inputs(d), quant=cfg.quant, act_scale_fmt=cfg.act_scale_fmt,
        w13_bias=None if b13 is None else np32(b13), w2_bias=None if b2 is None else np32(b2),
        router_weight_in_gemm2=in_gemm2, act_recipe=recipe, tokens=tokens, return_items=True)
    return y, flip_allowance(y, items, w)


CASES = {
    "bf16": (MoEConfig("ep16", M=300, H=512, I=256, E=8, topk=2, quant="bf16",
                       routing="softmax", seed=81), BF16_TOL),
    "fp8": (MoEConfig("ep8", M=200, H=512, I=256, E=8, topk=2, quant="fp8", routing="softmax",
                      seed=82, act_scale_fmt="ue8m0"), QUANT_TOL),
    "mxfp4": (MoEConfig("ep4", M=200, H=512, I=256, E=8, topk=2, quant="mxfp4",
                        routing="uniform", seed=83, act_scale_fmt="ue8m0"), QUANT_TOL),
}
VARIANTS = [  # (biases, router weight in GEMM2, recipe)
    (True, False, None), (False, True, None), (False, False, RECIPE), (True, True, RECIPE)]


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("bias,in_gemm2,recipe", VARIANTS)
def test_epilogue_variants(name, bias, in_gemm2, recipe):
    cfg, tol = CASES[name]
    d = make_inputs(cfg, "cuda")
    b13, b2 = _biases(cfg, 3) if bias else (None, None)
    p = moe.Problem.from_config(cfg, router_weight_in_gemm2=in_gemm2, act_recipe=recipe)
    forms = ["single", "pairs"] if cfg.quant == "bf16" else ["auto"]
    ref, allow = _oracle(cfg, d, b13, b2, in_gemm2, recipe)
    for form in forms:
        with bf16_gemm_form(form):
            y = _run(cfg, d, p, b13, b2)
        check_close(np32(y), ref, tol, f"{name} {form}", allow)


def test_router_weight_in_gemm2_stage_by_stage():
    """grouped_gemm_w2_ex with the router weight in its epilogue equals the
    oracle's weighted rows; unpermute_reduce then only sums."""
    cfg, _ = CASES["bf16"]
    d = make_inputs(cfg, "cuda")
    p = moe.Problem.from_config(cfg, router_weight_in_gemm2=True)
    b = moe.stage_buffers(p)
    moe.moe_align_permute(p, d["x"], d["topk_ids"], None, b["sorted_ids"], b["block_expert_ids"],
                          b["expert_offsets"], b["num_post_padded"], b["inv_perm"], b["x_perm"],
                          None, b["align_ws"])
    moe.grouped_gemm_w13(p, b["x_perm"], None, d["w13"], None, b["block_expert_ids"],
                         b["num_post_padded"], b["z"], None, fuse_act=True)
    moe.grouped_gemm_w2_ex(p, b["z"], None, d["w2"], None, None, b["block_expert_ids"],
                           b["num_post_padded"], b["sorted_ids"], d["topk_weights"], b["y2"])
    moe.unpermute_reduce(p, b["y2"], b["inv_perm"], None, b["y"])
    assert moe.moe_sync_status() == 0
    n = int(b["num_post_padded"].item())
    sid = b["sorted_ids"][:n].cpu().numpy()
    live = sid < cfg.M * cfg.topk
    # GEMM2 on the GPU's own z, weighted per row, against the GPU's y2
    a = oracle_inputs(d)
    route_ids = b["block_expert_ids"][: n // 128].cpu().numpy()
    zg = np32(b["z"])[:n].astype(np.float64)
    y2 = np.zeros((n, cfg.H))
    for blk, e in enumerate(route_ids):
        r = slice(blk * 128, blk * 128 + 128)
        y2[r] = zg[r] @ a["w2"][e].astype(np.float64).T
    wflat = a["topk_weights"].reshape(-1).astype(np.float64)
    y2 *= np.where(live, wflat[np.minimum(sid, cfg.M * cfg.topk - 1)], 0.0)[:, None]
    check_close(np32(b["y2"])[:n][live], codecs.round_bf16(y2[live]), BF16_TOL, "weighted y2")
    # the reduce sums the GPU's weighted rows with weight 1
    inv = b["inv_perm"].cpu().numpy()
    y2g = np32(b["y2"][:n]).astype(np.float64)      # rows past n hold no values
    want = np.zeros((cfg.M, cfg.H))
    for i in range(cfg.topk):
        ok = inv[:, i] >= 0
        want[ok] += y2g[inv[ok, i]]
    check_close(np32(b["y"]), codecs.round_bf16(want), BF16_TOL, "sum")


def test_variant_arguments_rejected():
    cfg, _ = CASES["bf16"]
    d = make_inputs(cfg, "cuda")
    p = moe.Problem.from_config(cfg, router_weight_in_gemm2=True)
    b = moe.stage_buffers(p)
    with pytest.raises(moe.MoEError) as ei:      # the plain GEMM2 entry has no weights
        moe.grouped_gemm_w2(p, b["z"], None, d["w2"], None, b["block_expert_ids"],
                            b["num_post_padded"], b["y2"])
    assert ei.value.status == 1
    q = moe.Problem.from_config(cfg.with_(topk=1), apply_router_weight_on_input=True,
                                router_weight_in_gemm2=True)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoEError) as ei:      # the weight is applied once
        moe.fused_experts(q, d["x"], d["w13"], None, d["w2"], None, d["topk_weights"][:, :1],
                          d["topk_ids"][:, :1].contiguous(), torch.empty_like(d["x"]), ws)
    assert ei.value.status == 1


@pytest.mark.parametrize("bias,in_gemm2,recipe", VARIANTS)
def test_fp8_fp32_scales_epilogue_stage_by_stage(bias, in_gemm2, recipe):
    """FP8 block scales with fp32 (not power-of-two) activation scales and
    every epilogue variant, stage by stage through the _ex entry points: each
    GPU stage against the oracle's same stage fed the GPU's own input (so a
    one-ulp difference upstream cannot move a group scale downstream), then
    the whole path against the oracle."""
    cfg = CASES["fp8"][0].with_(act_scale_fmt="fp32", seed=84)
    d = make_inputs(cfg, "cuda")
    b13, b2 = _biases(cfg, 5) if bias else (None, None)
    p = moe.Problem.from_config(cfg, router_weight_in_gemm2=in_gemm2, act_recipe=recipe)
    b = moe.stage_buffers(p)
    moe.moe_align_permute(p, d["x"], d["topk_ids"], None, b["sorted_ids"], b["block_expert_ids"],
                          b["expert_offsets"], b["num_post_padded"], b["inv_perm"], b["x_perm"],
                          b["x_perm_scale"], b["align_ws"])
    moe.grouped_gemm_w13_ex(p, b["x_perm"], b["x_perm_scale"], d["w13"], d["w13_scale"], b13,
                            b["block_expert_ids"], b["num_post_padded"], b["h1"], None,
                            fuse_act=False)
    moe.act_mul_quant(p, b["h1"], b["num_post_padded"], b["z"], b["z_scale"])
    moe.grouped_gemm_w2_ex(p, b["z"], b["z_scale"], d["w2"], d["w2_scale"], b2,
                           b["block_expert_ids"], b["num_post_padded"], b["sorted_ids"],
                           d["topk_weights"], b["y2"])
    moe.unpermute_reduce(p, b["y2"], b["inv_perm"], d["topk_weights"], b["y"])
    assert moe.moe_sync_status() == 0
    a = oracle_inputs(d)
    route = experts.align_permute(a["topk_ids"], cfg.E, 128)
    n = route["num_tokens_post_padded"]
    R = cfg.M * cfg.topk
    sid = route["sorted_token_ids"]
    live = sid[:n] < R
    xq, xs = experts.permute_rows(a["x"], route, cfg.topk, scale_fmt="fp32")
    # the quantising permute: codes and fp32 scales bit for bit
    assert np.array_equal(codecs.e4m3_decode(np32(b["x_perm"]))[:n][live], xq[:n][live])
    assert np.array_equal(np32(b["x_perm_scale"])[:n][live], xs[:n][live])
    h1 = experts.grouped_gemm(xq, xs, a["w13"], a["w13_scale"], route, 128, "fp8")
    h1 = experts.add_expert_bias(h1, None if b13 is None else np32(b13), route, 128)
    check_close(np32(b["h1"])[:n][live], codecs.round_bf16(h1[:n][live]), QUANT_TOL,
                "fp8 fp32-scale h1 (+bias)")
    # activation recipe + fp32 1x128 quantisation of the GPU's own h1
    h1g = np32(b["h1"]).astype(np.float64)
    zo, zso = experts.quant_act_1x128(experts.act_mul(h1g[:n], cfg.I, recipe=recipe), "fp32")
    zq = codecs.e4m3_decode(np32(b["z"])).astype(np.float64)
    zs = np32(b["z_scale"]).astype(np.float64)
    # scales: fp32 amax/448 on both sides, amax may differ in its last fp32 bit
    np.testing.assert_allclose(zs[:n][live], zso[live], rtol=2 ** -20)
    zg = zq[:n] * np.repeat(zs[:n], 128, axis=1)
    check_close(zg[live], (zo * np.repeat(zso, 128, axis=1))[live], QUANT_TOL,
                "fp8 fp32-scale z (recipe)" if recipe else "fp8 fp32-scale z")
    codes_equal = np.mean(np32(b["z"])[:n][live] == codecs.e4m3_encode(zo[live]))
    assert codes_equal > 0.999, codes_equal
    # GEMM2 (+bias, router weight) on the GPU's own z
    zq[n:] = 0
    zs[n:] = 0
    zq[:n][~live] = 0
    zs[:n][~live] = 0
    y2 = experts.grouped_gemm(zq, zs, a["w2"], a["w2_scale"], route, 128, "fp8")
    y2 = experts.add_expert_bias(y2, None if b2 is None else np32(b2), route, 128)
    if in_gemm2:
        wflat = a["topk_weights"].reshape(-1).astype(np.float64)
        y2 = y2 * np.where(sid < R, wflat[np.minimum(sid, R - 1)], 0.0)[:, None]
    check_close(np32(b["y2"])[:n][live], codecs.round_bf16(y2[:n][live]), QUANT_TOL,
                "fp8 fp32-scale y2")
    # the reduce of the GPU's y2
    y2g = np32(b["y2"]).astype(np.float64)
    want = experts.unpermute_reduce(y2g, route["inv_perm"], a["topk_weights"],
                                    apply_router_weight_on_input=in_gemm2)
    check_close(np32(b["y"]), want, QUANT_TOL, "fp8 fp32-scale reduce")
    # and the whole path against the oracle
    ref, allow = _oracle(cfg, d, b13, b2, in_gemm2, recipe)
    check_close(np32(b["y"]), ref, QUANT_TOL, "fp8 fp32-scale whole path", allow)
