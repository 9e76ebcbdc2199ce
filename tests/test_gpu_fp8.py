"""GPU parity of the FP8 path (e4m3 weights with fp32 128x128 block scales,
dynamic 1x128 activation quantisation): stage by stage on ragged expert loads
and end to end, including the DeepSeek-class workload at full size on sampled
tokens.  Tolerance 3e-2 * RMS (reading in gpu_util)."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import CONFIGS, MoEConfig, make_inputs
from oracle import codecs, experts, routing

from .gpu_util import (QUANT_TOL, bf16_gemm_form, check_close, cover_tokens, flip_allowance,
                       np32, oracle_inputs)

pytestmark = pytest.mark.gpu


def _fp8_ragged(counts, H, I, seed, fmt):
    E = len(counts)
    ids = np.concatenate([np.full(c, e, dtype=np.int32) for e, c in enumerate(counts)])
    np.random.default_rng(seed).shuffle(ids)
    M = len(ids)
    cfg = MoEConfig("r", M=M, H=H, I=I, E=E, topk=1, quant="fp8", routing="softmax", seed=seed,
                    act_scale_fmt=fmt)
    d = make_inputs(cfg, "cuda")
    d["topk_ids"] = torch.from_numpy(ids).view(M, 1).cuda()
    return cfg, d


@pytest.mark.parametrize("form", ["single", "pairs"])
@pytest.mark.parametrize("fmt", ["fp32", "ue8m0"])
@pytest.mark.parametrize("counts,H,I", [([0, 1, 127, 128, 129, 300], 512, 256),
                                        ([7, 0, 260], 384, 384),
                                        ([385, 0, 1, 640], 640, 384)])
def test_fp8_stages_ragged(counts, H, I, fmt, form):
    """Both GEMM forms (one SM; SM pairs, with lone and paired blocks and a
    128-wide last column tile at H = 640) on ragged expert loads."""
    with bf16_gemm_form(form):
        _fp8_stages_ragged(counts, H, I, fmt)


def _fp8_stages_ragged(counts, H, I, fmt):
    cfg, d = _fp8_ragged(counts, H, I, 5, fmt)
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
    xq, xs = experts.permute_rows(a["x"], route, 1, scale_fmt=fmt)
    # GEMM1 alone: the GPU's quantised x is bit-exact with the oracle's
    h1 = experts.grouped_gemm(xq, xs, a["w13"], a["w13_scale"], route, 128, "fp8")
    check_close(np32(b["h1"])[:n][live], codecs.round_bf16(h1[:n][live]), QUANT_TOL, "h1")
    # GEMM2 alone, on the GPU's own quantised z
    zq = codecs.e4m3_decode(np32(b["z"]))
    zs = np32(b["z_scale"]).astype(np.float64)
    zq[n:] = 0
    zs[n:] = 0
    y2 = experts.grouped_gemm(zq, zs, a["w2"], a["w2_scale"], route, 128, "fp8")
    check_close(np32(b["y2"])[:n][live], codecs.round_bf16(y2[:n][live]), QUANT_TOL, "y2")
    # whole path
    ref = experts.fused_experts(**a, quant="fp8", act_scale_fmt=fmt)
    inv = route["inv_perm"]
    items = np.where((inv >= 0)[..., None], ref["y2"][np.maximum(inv, 0)], 0.0)
    check_close(np32(b["y"]), ref["y"], QUANT_TOL, "y",
                allow=flip_allowance(ref["y"], items, a["topk_weights"]))


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


@pytest.mark.parametrize("form", ["auto", "single", "pairs"])
def test_fp8_fused_small_skewed(form):
    cfg = MoEConfig("fp8s", M=256, H=512, I=256, E=16, topk=4, quant="fp8", routing="skew",
                    seed=61)
    d = make_inputs(cfg, "cuda")
    with bf16_gemm_form(form):
        y = _run_fused(cfg, d)
    ref, allow = _oracle(cfg, d, range(cfg.M))
    check_close(np32(y), ref, QUANT_TOL, f"fp8 small {form}", allow)


def test_fp8_deepseek_full_size_sampled():
    cfg = CONFIGS["dsfp8"]
    d = make_inputs(cfg, "cuda")
    info = d["routing_info"]
    assert 0.49 <= info["hot_share"] <= 0.51, info
    y = _run_fused(cfg, d)
    yn = np32(y)
    assert np.all(np.isfinite(yn)) and np.all(np.abs(yn).max(axis=1) > 0)
    # every hot expert's first block, last block and last live row, and
    # random other tokens: 256 in all
    tokens = cover_tokens(d["topk_ids"], cfg.E, 256, 7, experts=range(info["hot_experts"]))
    assert len(tokens) >= 256
    ref, allow = _oracle(cfg, d, tokens)
    check_close(yn[tokens], ref, QUANT_TOL, f"dsfp8 full size, {len(tokens)} tokens", allow)
    assert torch.equal(_run_fused(cfg, d), y)
