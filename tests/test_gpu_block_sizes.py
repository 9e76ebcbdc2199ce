"""Block sizes 16, 32 and 64 through every stage (the validated set of the
pages' moe_align_block_size, page "fused_moe.py 分析", "moe_align_block_size
的作用"; the per-call alignment of page "Blackwell 上的 DeepGEMM FusedMoE（vLLM）",
§2.6.1).

The GEMMs cut each expert's padded segment into 128-row tiles; with a block
size below 128 the last tile of a segment is partial and its rows past the
segment belong to the next expert (or to no one): they must not be written.
Every routed item's row does the same arithmetic whatever the block size, so
the checks are bit for bit against block size 128: each routed item's H1, Z
(codes and scales), Y2 row and the whole output y; the whole path is also
checked against the oracle at one block size, and the rows of the padded
layout at or past num_tokens_post_padded are checked untouched."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import MoEConfig, make_inputs
from oracle import experts

from .gpu_util import BF16_TOL, QUANT_TOL, check_close, flip_allowance, np32, oracle_inputs

pytestmark = pytest.mark.gpu

COUNTS = [0, 1, 15, 16, 17, 63, 64, 65, 127, 128, 129, 300]
SENTINEL = 0x5A


def _inputs(quant, seed=41):
    ids = np.concatenate([np.full(c, e, dtype=np.int32) for e, c in enumerate(COUNTS)])
    np.random.default_rng(seed).shuffle(ids)
    M = len(ids)
    H = 512 if quant == "bf16" else 640
    fmt = "ue8m0" if quant in ("mxfp4", "mxfp8") else "fp32"
    cfg = MoEConfig("bs", M=M, H=H, I=256, E=len(COUNTS), topk=1, quant=quant,
                    routing="softmax", seed=seed, act_scale_fmt=fmt)
    d = make_inputs(cfg, "cuda")
    d["topk_ids"] = torch.from_numpy(ids).view(M, 1).cuda()
    return cfg, d


def _stages(cfg, d, bs, fuse):
    p = moe.Problem.from_config(cfg, block_size=bs)
    b = moe.stage_buffers(p)
    for k in ("x_perm", "h1", "z", "y2"):
        b[k].view(torch.uint8).fill_(SENTINEL)
    moe.moe_align_permute(p, d["x"], d["topk_ids"], None, b["sorted_ids"], b["block_expert_ids"],
                          b["expert_offsets"], b["num_post_padded"], b["inv_perm"], b["x_perm"],
                          b["x_perm_scale"], b["align_ws"])
    if fuse:
        moe.grouped_gemm_w13(p, b["x_perm"], b["x_perm_scale"], d["w13"], d["w13_scale"],
                             b["block_expert_ids"], b["num_post_padded"], b["z"], b["z_scale"],
                             fuse_act=True)
    else:
        moe.grouped_gemm_w13(p, b["x_perm"], b["x_perm_scale"], d["w13"], d["w13_scale"],
                             b["block_expert_ids"], b["num_post_padded"], b["h1"], None)
        moe.act_mul_quant(p, b["h1"], b["num_post_padded"], b["z"], b["z_scale"])
    moe.grouped_gemm_w2(p, b["z"], b["z_scale"], d["w2"], d["w2_scale"], b["block_expert_ids"],
                        b["num_post_padded"], b["y2"])
    moe.unpermute_reduce(p, b["y2"], b["inv_perm"], d["topk_weights"], b["y"])
    assert moe.moe_sync_status() == 0
    return b


@pytest.mark.parametrize("quant", ["bf16", "fp8", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("bs", [16, 32, 64])
@pytest.mark.parametrize("fuse", [False, True])
def test_stages_at_block_size_equal_block_128(quant, bs, fuse):
    cfg, d = _inputs(quant)
    ref = _stages(cfg, d, 128, fuse)
    got = _stages(cfg, d, bs, fuse)
    n = int(got["num_post_padded"].item())
    assert n % bs == 0
    inv_g = got["inv_perm"].view(-1).long()
    inv_r = ref["inv_perm"].view(-1).long()
    live = inv_g >= 0
    assert torch.equal(live, inv_r >= 0)
    keys = ["z", "y2"] + ([] if fuse else ["h1"]) + (["z_scale"] if quant != "bf16" else [])
    for k in keys:
        assert torch.equal(got[k][inv_g[live]], ref[k][inv_r[live]]), k
    assert torch.equal(got["y"], ref["y"])
    # nothing written at or past the used rows of the padded layout
    for k in ("x_perm", "y2", "z") + (() if fuse else ("h1",)):
        rest = got[k][n:].contiguous().view(torch.uint8)
        assert bool((rest == SENTINEL).all()), k


@pytest.mark.parametrize("quant", ["bf16", "fp8", "mxfp4", "mxfp8"])
def test_fused_experts_block_size_64_against_oracle(quant):
    cfg, d = _inputs(quant, seed=43)
    p64 = moe.Problem.from_config(cfg, block_size=64)
    p128 = moe.Problem.from_config(cfg)
    ys = []
    for p in (p64, p128):
        ws = torch.empty(moe.moe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
        y = torch.empty_like(d["x"])
        moe.fused_experts(p, d["x"], d["w13"], d["w13_scale"], d["w2"], d["w2_scale"],
                          d["topk_weights"], d["topk_ids"], y, ws)
        assert moe.moe_sync_status() == 0
        ys.append(y)
    assert torch.equal(ys[0], ys[1])
    ref, items, w = experts.fused_experts_per_token(
        **oracle_inputs(d), quant=cfg.quant, act_scale_fmt=cfg.act_scale_fmt, return_items=True)
    check_close(np32(ys[0]), ref, BF16_TOL if quant == "bf16" else QUANT_TOL,
                f"{quant} block size 64", flip_allowance(ref, items, w))
