"""GPU parity of stage 1 (block-aligned routing + permute) against the oracle:
indices bit-exact on every workload's routing and on edge cases; permuted
rows bit-exact (bf16 copy) and FP8 codes/scales bit-exact (both sides form
v / s in fp32 and round to e4m3 with ties to even)."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import CONFIGS, MoEConfig, make_inputs, make_routing
from oracle import codecs, experts, routing

from .gpu_util import np32

pytestmark = pytest.mark.gpu


def _run_routing(p, ids_dev, x=None, w=None):
    b = moe.stage_buffers(p)
    moe.moe_align_permute(p, x, ids_dev, w, b["sorted_ids"], b["block_expert_ids"],
                          b["expert_offsets"], b["num_post_padded"], b["inv_perm"],
                          b["x_perm"] if x is not None else None,
                          b["x_perm_scale"] if x is not None else None, b["align_ws"])
    assert moe.moe_sync_status() == 0
    return b


def _check_routing(b, ids_np, E, A):
    ref = routing.align_permute(ids_np, E, A)
    assert int(b["num_post_padded"].item()) == ref["num_tokens_post_padded"]
    assert np.array_equal(np32(b["expert_offsets"])[:E + 1], ref["expert_offsets"])
    assert np.array_equal(np32(b["sorted_ids"]), ref["sorted_token_ids"])
    assert np.array_equal(np32(b["block_expert_ids"]), ref["block_expert_ids"])
    assert np.array_equal(np32(b["inv_perm"]), ref["inv_perm"])
    return ref


@pytest.mark.parametrize("name", list(CONFIGS))
def test_routing_bit_exact_workloads(name):
    cfg = CONFIGS[name]
    w, ids, _ = make_routing(cfg, "cuda")
    p = moe.Problem.from_config(cfg)
    b = _run_routing(p, ids)
    _check_routing(b, np32(ids), cfg.E, cfg.block_size)


EDGE = [
    # (M, k, E, A, id generator)
    (1, 1, 1, 128, "all0"),
    (3, 2, 8, 16, "rand"),
    (513, 3, 5, 32, "rand"),          # R not a multiple of the 512-item segment
    (1000, 4, 1024, 64, "rand"),      # E at its maximum
    (2048, 8, 256, 128, "hot1"),      # one expert takes almost everything
    (700, 2, 16, 128, "invalid"),     # 40% of the slots are -1
    (64, 2, 64, 128, "invalid_all"),  # every slot skipped
    (16384, 1, 8, 128, "rand"),       # maximum token count
]


def _edge_ids(M, k, E, kind, seed=7):
    g = torch.Generator().manual_seed(seed)
    ids = torch.randint(0, E, (M, k), generator=g, dtype=torch.int32)
    if kind == "all0":
        ids.zero_()
    elif kind == "hot1":
        ids[torch.rand(M, k, generator=g) < 0.9] = 3
    elif kind == "invalid":
        ids[torch.rand(M, k, generator=g) < 0.4] = -1
    elif kind == "invalid_all":
        ids.fill_(-1)
    return ids


@pytest.mark.parametrize("M,k,E,A,kind", EDGE)
def test_routing_bit_exact_edge_cases(M, k, E, A, kind):
    ids = _edge_ids(M, k, E, kind)
    p = moe.Problem(M=M, H=128, I=128, E=E, topk=k, block_size=A)
    b = _run_routing(p, ids.cuda())
    _check_routing(b, ids.numpy(), E, A)


@pytest.mark.parametrize("M", [2, 8192])   # one-CTA small-batch form, three-kernel form
def test_routing_bad_index_reported(M):
    ids = torch.zeros(M, 2, dtype=torch.int32)
    ids[0] = torch.tensor([0, 1])
    ids[1] = torch.tensor([2, 8])
    p = moe.Problem(M=M, H=128, I=128, E=8, topk=2)
    b = moe.stage_buffers(p)
    moe.moe_align_permute(p, None, ids.cuda(), None, b["sorted_ids"], b["block_expert_ids"],
                          b["expert_offsets"], b["num_post_padded"], b["inv_perm"], None, None,
                          b["align_ws"])
    assert moe.moe_sync_status() == 6   # MOE_ERR_DEVICE_BAD_INDEX
    assert moe.moe_sync_status() == 0   # the error word was cleared
    # the bad slot is treated as skipped
    assert np32(b["inv_perm"])[1, 1] == -1


@pytest.mark.parametrize("name", ["tiny", "decode", "mixtral"])
def test_permute_bf16_bit_exact(name):
    cfg = CONFIGS[name]
    d = make_inputs(cfg, "cuda", weights=False)
    p = moe.Problem.from_config(cfg)
    b = _run_routing(p, d["topk_ids"], d["x"])
    ref = routing.align_permute(np32(d["topk_ids"]), cfg.E, cfg.block_size)
    n = ref["num_tokens_post_padded"]
    xp_ref, _ = experts.permute_rows(np32(d["x"]), ref, cfg.topk)
    assert np.array_equal(np32(b["x_perm"])[:n], xp_ref[:n])


def test_permute_router_weight_on_input_bit_exact():
    cfg = MoEConfig("arwoi", M=300, H=512, I=128, E=8, topk=1, quant="bf16", routing="softmax",
                    seed=31, apply_router_weight_on_input=True)
    d = make_inputs(cfg, "cuda", weights=False)
    p = moe.Problem.from_config(cfg)
    b = _run_routing(p, d["topk_ids"], d["x"], d["topk_weights"])
    ref = routing.align_permute(np32(d["topk_ids"]), cfg.E, cfg.block_size)
    n = ref["num_tokens_post_padded"]
    xp_ref, _ = experts.permute_rows(np32(d["x"]), ref, 1, np32(d["topk_weights"]))
    assert np.array_equal(np32(b["x_perm"])[:n], xp_ref[:n])


@pytest.mark.parametrize("name,fmt", [("dsfp8", "fp32"), ("dsfp8", "ue8m0"), ("mxfp4", "ue8m0")])
def test_permute_fp8_codes_bit_exact(name, fmt):
    cfg = CONFIGS[name].with_(act_scale_fmt=fmt)
    d = make_inputs(cfg, "cuda", weights=False)
    p = moe.Problem.from_config(cfg)
    b = _run_routing(p, d["topk_ids"], d["x"])
    ids = np32(d["topk_ids"])
    ref = routing.align_permute(ids, cfg.E, cfg.block_size)
    n = ref["num_tokens_post_padded"]
    R = cfg.M * cfg.topk
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.integers(0, n, 2000), np.arange(min(n, 300))]))
    sid = ref["sorted_token_ids"][rows]
    x = np32(d["x"]).astype(np.float64)
    live = sid < R
    src = np.where(live[:, None], x[np.minimum(sid, R - 1) // cfg.topk], 0.0)
    q, s = experts.quant_act_1x128(src, fmt)
    q[~live] = 0.0
    s[~live] = 0.0
    codes_gpu = np32(b["x_perm"])[rows]
    assert np.array_equal(codes_gpu, codecs.e4m3_encode(q))
    assert np.array_equal(np32(b["x_perm_scale"])[rows].astype(np.float64), s)


QPERM = [  # (M, k, E, H, kind, quant, fmt)
    (300, 3, 16, 384, "invalid", "fp8", "fp32"),      # 40% of the slots skipped, H/16 < 32 lanes
    (300, 3, 16, 384, "invalid", "mxfp8", "ue8m0"),
    (257, 8, 64, 1152, "rand", "fp8", "ue8m0"),       # top-8, ragged tail of 16-value chunks
    (257, 8, 64, 1152, "hot1", "mxfp8", "ue8m0"),     # one hot expert, many padded experts
    (64, 2, 64, 256, "invalid_all", "fp8", "fp32"),   # no routed row at all
    (1, 16, 32, 7168, "rand", "fp8", "fp32"),         # one token, the maximum top-k
]


@pytest.mark.parametrize("M,k,E,H,kind,quant,fmt", QPERM)
def test_permute_quant_every_row_bit_exact(M, k, E, H, kind, quant, fmt):
    """The quantising permute stores each token's codes into all of its routed
    rows and zeroes the padding rows: every row below num_post_padded is
    compared with the oracle (output buffers pre-filled with 0xFF so a row the
    kernel never writes shows up)."""
    ids = _edge_ids(M, k, E, kind, seed=M + k)
    g = torch.Generator().manual_seed(11)
    x = torch.randn(M, H, generator=g).to(torch.bfloat16)
    p = moe.Problem(M=M, H=H, I=128, E=E, topk=k, quant=quant, act_scale_fmt=fmt)
    b = moe.stage_buffers(p)
    b["x_perm"].fill_(0xFF)
    b["x_perm_scale"].fill_(float("nan"))
    moe.moe_align_permute(p, x.cuda(), ids.cuda(), None, b["sorted_ids"], b["block_expert_ids"],
                          b["expert_offsets"], b["num_post_padded"], b["inv_perm"], b["x_perm"],
                          b["x_perm_scale"], b["align_ws"])
    assert moe.moe_sync_status() == 0
    ref = _check_routing(b, ids.numpy(), E, 128)
    n = ref["num_tokens_post_padded"]
    q, s = experts.permute_rows(x.float().numpy(), ref, k, None, fmt, experts.act_group(quant))
    assert np.array_equal(np32(b["x_perm"])[:n], codecs.e4m3_encode(q[:n]))
    assert np.array_equal(np32(b["x_perm_scale"])[:n].astype(np.float64), s[:n])
