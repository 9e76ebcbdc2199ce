"""GEMM epilogue stores at both output alignments.

The epilogues write each output row 64 bytes at a time: as two 256-bit
stores where the row is 32-byte aligned, as four 16-byte stores otherwise
(the boundary only promises 16-byte aligned base addresses).  Both forms must
write the same bytes: every grouped GEMM runs once into a 32-byte aligned
buffer and once into a buffer 16 bytes past that, and the rows up to
num_tokens_post_padded are compared bit for bit."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import MoEConfig, make_inputs

from .gpu_util import bf16_gemm_form

pytestmark = pytest.mark.gpu

COUNTS = [0, 1, 127, 128, 129, 300]


def _inputs(quant, H, I):
    ids = np.concatenate([np.full(c, e, dtype=np.int32) for e, c in enumerate(COUNTS)])
    np.random.default_rng(21).shuffle(ids)
    M = len(ids)
    fmt = "fp32" if quant in ("bf16", "fp8") else "ue8m0"
    cfg = MoEConfig("align", M=M, H=H, I=I, E=len(COUNTS), topk=1, quant=quant,
                    routing="softmax", seed=21, act_scale_fmt=fmt)
    d = make_inputs(cfg, "cuda")
    d["topk_ids"] = torch.from_numpy(ids).view(M, 1).cuda()
    return cfg, d


def _shifted_like(t):
    """A tensor shaped like t whose data starts 16 bytes past a 32-byte boundary."""
    raw = torch.empty(t.numel() + 32, dtype=t.dtype, device=t.device)
    per = 16 // t.element_size()
    off = (-raw.data_ptr() % 32) // t.element_size() + per
    view = raw[off:off + t.numel()].view(t.shape)
    assert view.data_ptr() % 32 == 16
    return view


def _aligned_like(t):
    raw = torch.empty(t.numel() + 32, dtype=t.dtype, device=t.device)
    off = (-raw.data_ptr() % 32) // t.element_size()
    view = raw[off:off + t.numel()].view(t.shape)
    assert view.data_ptr() % 32 == 0
    return view


def _run(quant, H, I, fuse):
    cfg, d = _inputs(quant, H, I)
    p = moe.Problem.from_config(cfg)
    b = moe.stage_buffers(p)
    moe.moe_align_permute(p, d["x"], d["topk_ids"], None, b["sorted_ids"], b["block_expert_ids"],
                          b["expert_offsets"], b["num_post_padded"], b["inv_perm"], b["x_perm"],
                          b["x_perm_scale"], b["align_ws"])
    outs = {}
    for name, like in (("aligned", _aligned_like), ("shifted", _shifted_like)):
        h1 = like(b["h1"])
        y2 = like(b["y2"])
        if fuse:                      # bf16 only: SiLU-and-mul in the GEMM1 epilogue
            z = like(b["z"])
            moe.grouped_gemm_w13(p, b["x_perm"], None, d["w13"], None, b["block_expert_ids"],
                                 b["num_post_padded"], z, None, fuse_act=True)
            moe.grouped_gemm_w2(p, z, None, d["w2"], None, b["block_expert_ids"],
                                b["num_post_padded"], y2)
            outs[name] = (z, y2)
        else:
            moe.grouped_gemm_w13(p, b["x_perm"], b["x_perm_scale"], d["w13"], d["w13_scale"],
                                 b["block_expert_ids"], b["num_post_padded"], h1)
            moe.act_mul_quant(p, h1, b["num_post_padded"], b["z"], b["z_scale"])
            moe.grouped_gemm_w2(p, b["z"], b["z_scale"], d["w2"], d["w2_scale"],
                                b["block_expert_ids"], b["num_post_padded"], y2)
            outs[name] = (h1, y2)
    assert moe.moe_sync_status() == 0
    n = int(b["num_post_padded"].item())
    assert n > 0
    for a, s in zip(outs["aligned"], outs["shifted"]):
        assert torch.equal(a[:n].view(torch.int16), s[:n].view(torch.int16))


@pytest.mark.parametrize("form", ["single", "pairs"])
@pytest.mark.parametrize("fuse", [False, True])
def test_bf16_epilogue_stores_at_both_alignments(form, fuse):
    with bf16_gemm_form(form):
        _run("bf16", 512, 256, fuse)


@pytest.mark.parametrize("quant", ["fp8", "mxfp4", "mxfp8"])
def test_quantised_epilogue_stores_at_both_alignments(quant):
    # H = 640: GEMM2's last column tile is 128 wide (N % 256 == 128)
    _run(quant, 640, 256, False)


def test_fp8_pair_epilogue_stores_at_both_alignments():
    with bf16_gemm_form("pairs"):
        _run("fp8", 640, 256, False)
