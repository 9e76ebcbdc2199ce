"""GPU parity of the MXFP4 W4A8 path (E2M1 weights with E8M0 scales per 32
along K, e4m3 activations with UE8M0 1x128 scales, block-scaled tensor-core
MMA): stage by stage on ragged expert loads, end to end on a small layer and
on the DeepSeek-class MXFP4 workload at full size (sampled tokens).
Tolerance 3e-2 * RMS (reading in gpu_util)."""
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
    cfg = MoEConfig("mx_r", M=M, H=H, I=I, E=E, topk=1, quant="mxfp4", routing="uniform",
                    seed=seed, act_scale_fmt="ue8m0")
    d = make_inputs(cfg, "cuda")
    d["topk_ids"] = torch.from_numpy(ids).view(M, 1).cuda()
    return cfg, d


@pytest.mark.parametrize("counts,H,I", [([0, 1, 127, 128, 129, 300], 512, 256),
                                        ([7, 0, 260], 384, 384),
                                        # K % 512 == 0: weight scales staged by TMA (GEMM2
                                        # here, with a ragged last column tile, N = 640)
                                        ([0, 1, 127, 128, 129, 300], 640, 512),
                                        ([5, 200, 0, 131], 1024, 512)])
def test_mxfp4_stages_ragged(counts, H, I):
    cfg, d = _ragged(counts, H, I, 9)
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
    xq, xs = experts.permute_rows(a["x"], route, 1, scale_fmt="ue8m0")
    h1 = experts.grouped_gemm(xq, xs, a["w13"], a["w13_scale"], route, 128, "mxfp4")
    check_close(np32(b["h1"])[:n][live], codecs.round_bf16(h1[:n][live]), QUANT_TOL, "h1")
    zq = codecs.e4m3_decode(np32(b["z"]))
    zs = np32(b["z_scale"]).astype(np.float64)
    zq[n:] = 0
    zs[n:] = 0
    y2 = experts.grouped_gemm(zq, zs, a["w2"], a["w2_scale"], route, 128, "mxfp4")
    check_close(np32(b["y2"])[:n][live], codecs.round_bf16(y2[:n][live]), QUANT_TOL, "y2")
    ref = experts.fused_experts(**a, quant="mxfp4", act_scale_fmt="ue8m0")
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


def test_mxfp4_fused_small():
    cfg = MoEConfig("mxs", M=200, H=512, I=256, E=16, topk=4, quant="mxfp4", routing="uniform",
                    seed=91, act_scale_fmt="ue8m0")
    d = make_inputs(cfg, "cuda")
    y = _run_fused(cfg, d)
    ref, allow = _oracle(cfg, d, range(cfg.M))
    check_close(np32(y), ref, QUANT_TOL, "mxfp4 small", allow)


def test_mxfp4_requires_power_of_two_activation_scales():
    cfg = MoEConfig("mxf", M=8, H=256, I=128, E=2, topk=1, quant="mxfp4", routing="uniform",
                    seed=92, act_scale_fmt="fp32")
    d = make_inputs(cfg, "cuda")
    with pytest.raises(moe.MoEError) as ei:
        _run_fused(cfg, d)
    assert ei.value.status == 2   # MOE_ERR_UNSUPPORTED


def test_mxfp4_deepseek_full_size_sampled():
    cfg = CONFIGS["mxfp4"]
    d = make_inputs(cfg, "cuda")
    y = _run_fused(cfg, d)
    yn = np32(y)
    assert np.all(np.isfinite(yn)) and np.all(np.abs(yn).max(axis=1) > 0)
    # uniform routing: the last live row of every expert (the edge of its
    # partial block), then random other tokens up to 256
    tokens = cover_tokens(d["topk_ids"], cfg.E, 256, 8, which=("last",))
    assert len(tokens) >= 256
    ref, allow = _oracle(cfg, d, tokens)
    check_close(yn[tokens], ref, QUANT_TOL, f"mxfp4 full size, {len(tokens)} tokens", allow)
    assert torch.equal(_run_fused(cfg, d), y)
