"""moe_prepack_weights: the load-time rewrite of the MXFP4 / MXFP8 weight
scales into the operand layout of the block-scaled MMA (page "Blackwell 上的
DeepGEMM FusedMoE（vLLM）", §2.8, transform_sf_into_required_layout).

The packed bytes are checked against the layout the header states, rebuilt
here with numpy; the GEMMs and fused_experts fed the packed scales must give
the unpacked calls' results bit for bit (the MMA reads the same operands), on
ragged expert loads, both GEMM1 forms (fused activation or not), a 128-wide
last column tile, K with and without the staged-scale form (K % 512), and the
MXFP4 workload at full size."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import CONFIGS, MoEConfig, make_inputs

from .gpu_util import bf16_gemm_form, np32

pytestmark = pytest.mark.gpu


def _pack_reference(scale):
    """[E, N, K/32] bytes -> [E][K/128][N/128] blocks of 512 bytes, block byte
    16 l + 4 c + j = scale[e, 128 g + 32 c + l, 4 kb + j]."""
    E, N, KQ = scale.shape
    G, KB = N // 128, KQ // 4
    s = scale.reshape(E, G, 4, 32, KB, 4)                # e, g, c, l, kb, j
    return np.ascontiguousarray(s.transpose(0, 4, 1, 3, 2, 5)).reshape(-1)   # e kb g l c j


def _packed(p, d):
    a = torch.empty(moe.moe_prepacked_scale_bytes(p, 0), dtype=torch.uint8, device="cuda")
    b = torch.empty(moe.moe_prepacked_scale_bytes(p, 1), dtype=torch.uint8, device="cuda")
    moe.moe_prepack_weights(p, d["w13_scale"], d["w2_scale"], a, b)
    assert moe.moe_sync_status() == 0
    return a, b


def _ragged(quant, counts, H, I, seed):
    ids = np.concatenate([np.full(c, e, dtype=np.int32) for e, c in enumerate(counts)])
    np.random.default_rng(seed).shuffle(ids)
    M = len(ids)
    cfg = MoEConfig("pk", M=M, H=H, I=I, E=len(counts), topk=1, quant=quant,
                    routing="uniform", seed=seed, act_scale_fmt="ue8m0")
    d = make_inputs(cfg, "cuda")
    d["topk_ids"] = torch.from_numpy(ids).view(M, 1).cuda()
    return cfg, d


@pytest.mark.parametrize("quant", ["mxfp4", "mxfp8"])
def test_packed_layout_bytes(quant):
    cfg = MoEConfig("pkl", M=8, H=640, I=384, E=3, topk=1, quant=quant, routing="uniform",
                    seed=5, act_scale_fmt="ue8m0")
    d = make_inputs(cfg, "cuda")
    p = moe.Problem.from_config(cfg)
    a, b = _packed(p, d)
    assert np.array_equal(np32(a), _pack_reference(np32(d["w13_scale"])))
    assert np.array_equal(np32(b), _pack_reference(np32(d["w2_scale"])))


def _stages(p, d, w13s, w2s, fuse):
    b = moe.stage_buffers(p)
    moe.moe_align_permute(p, d["x"], d["topk_ids"], None, b["sorted_ids"], b["block_expert_ids"],
                          b["expert_offsets"], b["num_post_padded"], b["inv_perm"], b["x_perm"],
                          b["x_perm_scale"], b["align_ws"])
    if fuse:
        moe.grouped_gemm_w13(p, b["x_perm"], b["x_perm_scale"], d["w13"], w13s,
                             b["block_expert_ids"], b["num_post_padded"], b["z"], b["z_scale"],
                             fuse_act=True)
    else:
        moe.grouped_gemm_w13(p, b["x_perm"], b["x_perm_scale"], d["w13"], w13s,
                             b["block_expert_ids"], b["num_post_padded"], b["h1"], None)
        moe.act_mul_quant(p, b["h1"], b["num_post_padded"], b["z"], b["z_scale"])
    moe.grouped_gemm_w2(p, b["z"], b["z_scale"], d["w2"], w2s, b["block_expert_ids"],
                        b["num_post_padded"], b["y2"])
    moe.unpermute_reduce(p, b["y2"], b["inv_perm"], d["topk_weights"], b["y"])
    assert moe.moe_sync_status() == 0
    return b


@pytest.mark.parametrize("quant", ["mxfp4", "mxfp8"])
@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("counts,H,I", [([0, 1, 127, 128, 129, 300], 640, 256),
                                        ([7, 0, 260], 1024, 512),
                                        ([256, 384, 5, 128], 1024, 256)])
@pytest.mark.parametrize("form", ["auto", "pairs"])
def test_prepacked_stages_equal_unpacked(quant, fuse, counts, H, I, form):
    """Both forms of the block-scaled GEMM on prepacked scales (one SM, and SM
    pairs: lone and paired blocks, a 128-wide last column tile) against the
    single-SM GEMM on the scales as given, bit for bit."""
    cfg, d = _ragged(quant, counts, H, I, 17)
    p = moe.Problem.from_config(cfg)
    pp = moe.Problem.from_config(cfg, weight_scales_prepacked=True)
    a, b = _packed(p, d)
    ref = _stages(p, d, d["w13_scale"], d["w2_scale"], fuse)
    with bf16_gemm_form(form):
        got = _stages(pp, d, a, b, fuse)
    n = int(ref["num_post_padded"].item())
    keys = ("z", "z_scale", "y2") if fuse else ("h1", "z", "z_scale", "y2")
    for k in keys:
        assert torch.equal(got[k][:n], ref[k][:n]), k
    assert torch.equal(got["y"], ref["y"])


def test_prepacked_fused_experts_full_size():
    cfg = CONFIGS["mxfp4"]
    d = make_inputs(cfg, "cuda")
    p = moe.Problem.from_config(cfg)
    pp = moe.Problem.from_config(cfg, weight_scales_prepacked=True)
    a, b = _packed(p, d)
    ws = torch.empty(moe.moe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    y_ref, y = torch.empty_like(d["x"]), torch.empty_like(d["x"])
    moe.fused_experts(p, d["x"], d["w13"], d["w13_scale"], d["w2"], d["w2_scale"],
                      d["topk_weights"], d["topk_ids"], y_ref, ws)
    moe.fused_experts(pp, d["x"], d["w13"], a, d["w2"], b, d["topk_weights"], d["topk_ids"], y,
                      ws)
    assert moe.moe_sync_status() == 0
    assert torch.equal(y, y_ref)


def test_prepack_rejects_other_modes():
    cfg = MoEConfig("pkr", M=8, H=256, I=128, E=2, topk=1, quant="fp8", routing="uniform",
                    seed=6)
    d = make_inputs(cfg, "cuda")
    p = moe.Problem.from_config(cfg)
    buf = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_prepack_weights(p, d["w13_scale"], d["w2_scale"], buf, buf)
    assert ei.value.status == 2                    # MOE_ERR_UNSUPPORTED
    assert moe.moe_prepacked_scale_bytes(p, 0) == 0
    # the flag belongs to the MX modes: any other mode is an invalid problem
    q = moe.Problem.from_config(cfg, weight_scales_prepacked=True)
    assert moe.moe_m_sum_bound(q) == 0
    with pytest.raises(moe.MoEError) as ei:
        moe.fused_experts(q, d["x"], d["w13"], d["w13_scale"], d["w2"], d["w2_scale"],
                          d["topk_weights"], d["topk_ids"], torch.empty_like(d["x"]), buf)
    assert ei.value.status == 1                    # MOE_ERR_INVALID_ARG
