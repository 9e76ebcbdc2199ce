"""GPU parity of the MXFP8 (1x32) recipe: e4m3 weights with E8M0 scales per
1x32, activations quantised per 1x32 with UE8M0 scales.  Stage by stage on
ragged expert loads (both scale-writer forms: K % 512 == 0 stages the weight
scales by TMA, other K loads them per lane; a ragged last column tile), the
fused path on a small case, and the DeepSeek-class shape at full size on
sampled tokens."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import CONFIGS, MoEConfig, make_inputs
from oracle import codecs, experts, routing

from .gpu_util import QUANT_TOL, check_close, cover_tokens, flip_allowance, np32, oracle_inputs

pytestmark = pytest.mark.gpu


def _ragged(counts, H, I, seed):
    E = len(counts)
    ids = np.concatenate([np.full(c, e, dtype=np.int32) for e, c in enumerate(counts)])
    np.random.default_rng(seed).shuffle(ids)
    M = len(ids)
    cfg = MoEConfig("m8r", M=M, H=H, I=I, E=E, topk=1, quant="mxfp8", routing="uniform",
                    seed=seed, act_scale_fmt="ue8m0")
    d = make_inputs(cfg, "cuda")
    d["topk_ids"] = torch.from_numpy(ids).view(M, 1).cuda()
    return cfg, d


@pytest.mark.parametrize("counts,H,I", [([0, 1, 127, 128, 129, 300], 512, 256),
                                        ([0, 1, 127, 128, 129, 300], 640, 512),
                                        ([7, 0, 260], 384, 384)])
def test_mxfp8_stages_ragged(counts, H, I):
    cfg, d = _ragged(counts, H, I, 21)
    p = moe.Problem.from_config(cfg)
    b = moe.stage_buffers(p)
    moe.moe_align_permute(p, d["x"], d["topk_ids"], None, b["sorted_ids"], b["block_expert_ids"],
                          b["expert_offsets"], b["num_post_padded"], b["inv_perm"], b["x_perm"],
                          b["x_perm_scale"], b["align_ws"])
    moe.grouped_gemm_w13(p, b["x_perm"], b["x_perm_scale"], d["w13"], d["w13_scale"],
                         b["block_expert_ids"], b["num_post_padded"], b["h1"])
    moe.act_mul_quant(p, b["h1"], b["num_post_padded"], b["z"], b["z_scale"])
    moe.grouped_gemm_w2(p, b["z"], b["z_scale"], d["w2"], d["w2_scale"], b["block_expert_ids"],
                        b["num_post_padded"], b["y2"])
    moe.unpermute_reduce(p, b["y2"], b["inv_perm"], d["topk_weights"], b["y"])
    assert moe.moe_sync_status() == 0
    a = oracle_inputs(d)
    route = routing.align_permute(a["topk_ids"], cfg.E, 128)
    n = route["num_tokens_post_padded"]
    live = route["sorted_token_ids"][:n] < cfg.M
    # stage 1: 1x32 codes and UE8M0 scales bit for bit
    xq, xs = experts.permute_rows(a["x"], route, 1, scale_fmt="ue8m0", group=32)
    assert np.array_equal(codecs.e4m3_decode(np32(b["x_perm"])[:n]), xq[:n])
    assert np.array_equal(np32(b["x_perm_scale"])[:n].astype(np.float64), xs[:n])
    # GEMM1 on identical quantised inputs
    h1 = experts.grouped_gemm(xq, xs, a["w13"], a["w13_scale"], route, 128, "mxfp8")
    check_close(np32(b["h1"])[:n][live], codecs.round_bf16(h1[:n][live]), QUANT_TOL, "h1")
    # stage 3 on the GPU's own h1: codes and scales bit for bit
    zq, zs = experts.quant_act_1x128(
        experts.act_mul(np32(b["h1"])[:n], cfg.I), "ue8m0", 32)
    gz, gs = codecs.e4m3_decode(np32(b["z"])[:n]), np32(b["z_scale"])[:n].astype(np.float64)
    agree = np.mean(gz[live] == zq[live])
    assert agree > 0.999, agree           # SiLU's fast exp may move a code at a rounding tie
    # GEMM2 on the GPU's own quantised z
    zq2 = np.zeros((len(route["sorted_token_ids"]), cfg.I))
    zs2 = np.zeros((len(route["sorted_token_ids"]), cfg.I // 32))
    zq2[:n], zs2[:n] = gz, gs
    zq2[:n][~live] = 0
    zs2[:n][~live] = 0
    y2 = experts.grouped_gemm(zq2, zs2, a["w2"], a["w2_scale"], route, 128, "mxfp8")
    check_close(np32(b["y2"])[:n][live], codecs.round_bf16(y2[:n][live]), QUANT_TOL, "y2")


def _run_fused(cfg, d):
    p = moe.Problem.from_config(cfg)
    ws = torch.empty(moe.moe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(d["x"])
    moe.fused_experts(p, d["x"], d["w13"], d["w13_scale"], d["w2"], d["w2_scale"],
                      d["topk_weights"], d["topk_ids"], y, ws)
    assert moe.moe_sync_status() == 0
    return y


def _oracle(cfg, d, tokens):
    y, items, w = experts.fused_experts_per_token(
        **oracle_inputs(d), quant=cfg.quant, act_scale_fmt=cfg.act_scale_fmt, tokens=tokens,
        return_items=True)
    return y, flip_allowance(y, items, w)


def test_mxfp8_fused_small():
    cfg = MoEConfig("m8s", M=200, H=512, I=512, E=16, topk=4, quant="mxfp8", routing="uniform",
                    seed=22, act_scale_fmt="ue8m0")
    d = make_inputs(cfg, "cuda")
    y = _run_fused(cfg, d)
    ref, allow = _oracle(cfg, d, range(cfg.M))
    check_close(np32(y), ref, QUANT_TOL, "mxfp8 small", allow)


def test_mxfp8_full_size_sampled():
    cfg = CONFIGS["mxfp8"]
    d = make_inputs(cfg, "cuda")
    y = _run_fused(cfg, d)
    yn = np32(y)
    assert np.all(np.isfinite(yn)) and np.all(np.abs(yn).max(axis=1) > 0)
    tokens = cover_tokens(d["topk_ids"], cfg.E, 256, 9,
                          experts=range(d["routing_info"]["hot_experts"]))
    assert len(tokens) >= 256
    ref, allow = _oracle(cfg, d, tokens)
    check_close(yn[tokens], ref, QUANT_TOL, f"mxfp8 full size, {len(tokens)} tokens", allow)
    assert torch.equal(_run_fused(cfg, d), y)


def test_mxfp8_requires_power_of_two_activation_scales():
    cfg = MoEConfig("m8f", M=8, H=256, I=128, E=2, topk=1, quant="mxfp8", routing="uniform",
                    seed=23, act_scale_fmt="fp32")
    d = make_inputs(cfg, "cuda")
    with pytest.raises(moe.MoEError) as ei:
        _run_fused(cfg, d)
    assert ei.value.status == 2   # MOE_ERR_UNSUPPORTED
