"""GPU parity of the router (moe_topk_router) against the oracle: selected
ids and token-expert indices bit-exact, weights within WEIGHT_RTOL; shapes
from one token to the boundary's M limit, E from 1 to 1024 (not a multiple of
32 included), k up to 16, fp32 and bf16 logits, tie-heavy integer logits,
softmax and sigmoid, with and without renormalisation, the pages' expert-map
example, and the router feeding the fused path."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import MoEConfig, make_inputs
from oracle import experts, router

from .gpu_util import BF16_TOL, check_close, flip_allowance, np32

pytestmark = pytest.mark.gpu

# fp32 weights: expf is within 2 ulp, each weight takes one division and its
# denominator at most ~40 fp32 roundings (a lane's 32 terms + 5 warp steps),
# so the relative error stays below 40 * 2^-24 ~ 2.4e-6; 1e-5 leaves room.
WEIGHT_RTOL = 1e-5


def _gpu_router(x, k, scoring, renorm, emap=None):
    M = x.shape[0]
    w = torch.empty(M, k, dtype=torch.float32, device="cuda")
    ids = torch.empty(M, k, dtype=torch.int32, device="cuda")
    tei = torch.empty(M, k, dtype=torch.int32, device="cuda")
    moe.moe_topk_router(x, k, w, ids, tei, scoring=scoring, renormalize=renorm,
                        expert_map=emap)
    assert moe.moe_sync_status() == 0
    return w.cpu().numpy(), ids.cpu().numpy(), tei.cpu().numpy()


def _logits(M, E, dtype, seed, ties=False):
    g = torch.Generator().manual_seed(seed)
    if ties:
        x = torch.randint(-3, 4, (M, E), generator=g).float()
    else:
        x = torch.randn(M, E, generator=g) * 2
    return x.to(dtype).cuda()


SHAPES = [(1, 8, 2), (333, 8, 2), (1000, 64, 6), (517, 256, 8), (64, 1000, 16), (257, 33, 16),
          (100, 1, 1), (50, 1024, 16), (16384, 256, 8)]


@pytest.mark.parametrize("M,E,k", SHAPES)
@pytest.mark.parametrize("scoring", ["softmax", "sigmoid"])
def test_router_matches_oracle(M, E, k, scoring):
    for dtype, renorm, seed in ((torch.float32, True, 1), (torch.bfloat16, False, 2)):
        x = _logits(M, E, dtype, seed)
        w, ids, tei = _gpu_router(x, k, scoring, renorm)
        rw, rids, rtei = router.topk_router(x.float().cpu().numpy(), k, renorm, scoring)
        np.testing.assert_array_equal(ids, rids)
        np.testing.assert_array_equal(tei, rtei)
        np.testing.assert_allclose(w, rw, rtol=WEIGHT_RTOL, atol=0)


@pytest.mark.parametrize("E,k", [(8, 8), (64, 16), (300, 5)])
def test_router_ties_resolve_to_lower_expert(E, k):
    x = _logits(777, E, torch.float32, 5, ties=True)
    w, ids, _ = _gpu_router(x, k, "softmax", True)
    rw, rids, _ = router.topk_router(x.cpu().numpy(), k, True, "softmax")
    np.testing.assert_array_equal(ids, rids)
    np.testing.assert_allclose(w, rw, rtol=WEIGHT_RTOL, atol=0)


def test_router_signed_zeros_tie():
    """-0 and +0 compare equal, so the lower expert wins between them."""
    x = torch.zeros(64, 40)
    x[:, 1::2] = -0.0
    x[:, 7] = 1.0
    x = x.cuda()
    w, ids, _ = _gpu_router(x, 6, "softmax", True)
    rw, rids, _ = router.topk_router(x.cpu().numpy(), 6, True, "softmax")
    np.testing.assert_array_equal(ids, rids)
    np.testing.assert_allclose(w, rw, rtol=WEIGHT_RTOL, atol=0)


def test_router_expert_map(golden_dir):
    import json
    import os
    with open(os.path.join(golden_dir, "router_hand_worked.json")) as f:
        g = json.load(f)["expert_map"]
    emap = np.array(g["map"], dtype=np.int32)
    x = _logits(400, len(emap), torch.float32, 7)
    em = torch.from_numpy(emap).cuda()
    w, ids, _ = _gpu_router(x, 2, "softmax", True, em)
    rw, rids, _ = router.topk_router(x.cpu().numpy(), 2, True, "softmax", expert_map=emap)
    np.testing.assert_array_equal(ids, rids)
    np.testing.assert_allclose(w, rw, rtol=WEIGHT_RTOL, atol=0)
    # a random shard map over 256 experts (a quarter local)
    rng = np.random.default_rng(3)
    emap = np.full(256, -1, np.int32)
    local = rng.choice(256, 64, replace=False)
    emap[local] = np.arange(64, dtype=np.int32)
    x = _logits(999, 256, torch.bfloat16, 8)
    w, ids, _ = _gpu_router(x, 8, "sigmoid", True, torch.from_numpy(emap).cuda())
    rw, rids, _ = router.topk_router(x.float().cpu().numpy(), 8, True, "sigmoid",
                                     expert_map=emap)
    np.testing.assert_array_equal(ids, rids)
    np.testing.assert_allclose(w, rw, rtol=WEIGHT_RTOL, atol=0)


def test_router_feeds_the_fused_path():
    """Logits -> router -> fused_experts on the GPU equals the oracle's router
    followed by the oracle's per-token forward."""
    cfg = MoEConfig("rt", M=300, H=512, I=256, E=16, topk=4, quant="bf16", routing="softmax",
                    seed=61)
    d = make_inputs(cfg, "cuda", weights=True)
    logits = _logits(cfg.M, cfg.E, torch.float32, 9)
    w = torch.empty(cfg.M, cfg.topk, dtype=torch.float32, device="cuda")
    ids = torch.empty(cfg.M, cfg.topk, dtype=torch.int32, device="cuda")
    moe.moe_topk_router(logits, cfg.topk, w, ids)
    p = moe.Problem.from_config(cfg)
    ws = torch.empty(moe.moe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(d["x"])
    moe.fused_experts(p, d["x"], d["w13"], None, d["w2"], None, w, ids, y, ws)
    assert moe.moe_sync_status() == 0
    rw, rids, _ = router.topk_router(logits.cpu().numpy(), cfg.topk, True, "softmax")
    np.testing.assert_array_equal(ids.cpu().numpy(), rids)
    ref, items, wts = experts.fused_experts_per_token(
        np32(d["x"]).astype(np.float64), rids, rw, np32(d["w13"]).astype(np.float64),
        np32(d["w2"]).astype(np.float64), return_items=True)
    check_close(np32(y), ref, BF16_TOL, "router+path", flip_allowance(ref, items, wts))
