"""GPU parity of the whole forward (fused_experts through the C ABI) against
the oracle, at the workloads' full sizes where the oracle can follow (tiny,
decode: every token; Mixtral-shaped prefill: sampled tokens, whose outputs the
per-token oracle computes one by one, plus size-independent properties of the
full output), and on edge cases: skipped slots, in-place output, host-buffer
entry, top-1 with the router weight applied on the input, a dense E = 1 case
and one token."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import CONFIGS, MoEConfig, make_inputs
from oracle import experts

from .gpu_util import (BF16_TOL, bf16_gemm_form, check_close, cover_tokens, flip_allowance,
                       np32, oracle_inputs)

pytestmark = pytest.mark.gpu


def _run(cfg, d, inplace=False):
    p = moe.Problem.from_config(cfg)
    ws = torch.empty(moe.moe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    x = d["x"].clone() if inplace else d["x"]
    y = x if inplace else torch.empty_like(d["x"])
    moe.fused_experts(p, x, d["w13"], d["w13_scale"], d["w2"], d["w2_scale"],
                      d["topk_weights"], d["topk_ids"], y, ws)
    assert moe.moe_sync_status() == 0
    return y


def _oracle_tokens(cfg, d, tokens):
    """Per-token oracle for ``tokens``: (y_ref, flip allowance)."""
    a = oracle_inputs(d)
    y, items, w = experts.fused_experts_per_token(
        **a, quant=cfg.quant, act_scale_fmt=cfg.act_scale_fmt,
        apply_router_weight_on_input=cfg.apply_router_weight_on_input, tokens=tokens,
        return_items=True)
    return y, flip_allowance(y, items, w)


SMALL_CASES = {
    "tiny": CONFIGS["tiny"],
    "decode": CONFIGS["decode"],
    "invalid_slots": MoEConfig("inv", M=200, H=512, I=256, E=8, topk=3, quant="bf16",
                               routing="softmax", seed=41, invalid_frac=0.25),
    "one_token": MoEConfig("one", M=1, H=256, I=128, E=8, topk=2, quant="bf16",
                           routing="softmax", seed=42),
    "dense_E1": MoEConfig("dense", M=130, H=256, I=256, E=1, topk=1, quant="bf16",
                          routing="softmax", seed=43),
    "top1_weight_on_input": MoEConfig("arwoi", M=150, H=512, I=256, E=4, topk=1,
                                      quant="bf16", routing="softmax", seed=44,
                                      apply_router_weight_on_input=True),
    "many_experts": MoEConfig("e64", M=96, H=256, I=128, E=64, topk=6, quant="bf16",
                              routing="softmax", seed=45),
}


@pytest.mark.parametrize("name", list(SMALL_CASES))
@pytest.mark.parametrize("form", ["auto", "pairs"])
def test_fused_experts_all_tokens(name, form):
    """At these sizes "auto" picks the single-SM GEMMs; "pairs" puts lone and
    odd blocks, skipped slots and one-block experts through the pair form."""
    cfg = SMALL_CASES[name]
    d = make_inputs(cfg, "cuda")
    with bf16_gemm_form(form):
        y = _run(cfg, d)
    ref, allow = _oracle_tokens(cfg, d, range(cfg.M))
    check_close(np32(y), ref, BF16_TOL, name, allow)
    if name == "tiny":
        # the permuted oracle gives the same answer
        ref2 = experts.fused_experts(**oracle_inputs(d))["y"]
        check_close(np32(y), ref2, BF16_TOL, name, allow)


def test_fused_experts_inplace_and_host_entry():
    cfg = CONFIGS["tiny"].with_(M=300, seed=51)
    d = make_inputs(cfg, "cuda")
    y = _run(cfg, d)
    y_in = _run(cfg, d, inplace=True)
    assert torch.equal(y, y_in)
    p = moe.Problem.from_config(cfg)
    ws = torch.empty(moe.moe_host_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    hx = d["x"].cpu().pin_memory()
    hid = d["topk_ids"].cpu().pin_memory()
    hw = d["topk_weights"].cpu().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    moe.fused_experts_from_host(p, hx, hid, hw, hy, d["w13"], None, d["w2"], None, ws)
    assert moe.moe_sync_status() == 0
    assert torch.equal(hy, y.cpu())
    # pageable host buffers take the staged-copy path; a pinned x with a
    # pageable y mixes the two
    px, py = d["x"].cpu(), torch.zeros_like(hx)
    moe.fused_experts_from_host(p, px, hid, hw, py, d["w13"], None, d["w2"], None, ws)
    assert moe.moe_sync_status() == 0
    assert torch.equal(py, y.cpu())
    py2 = torch.zeros_like(hx)
    moe.fused_experts_from_host(p, hx, hid, hw, py2, d["w13"], None, d["w2"], None, ws)
    assert moe.moe_sync_status() == 0
    assert torch.equal(py2, y.cpu())


@pytest.mark.parametrize("name", ["mixtral"])
@pytest.mark.parametrize("form", ["auto", "single"])
def test_fused_experts_full_size_sampled(name, form):
    """"auto" is the pair form at this size (the benchmarked launch)."""
    cfg = CONFIGS[name]
    d = make_inputs(cfg, "cuda")
    with bf16_gemm_form(form):
        y = _run(cfg, d)
        y_again = _run(cfg, d)
    yn = np32(y)
    # properties at full size: finite, non-trivial, every token written
    assert np.all(np.isfinite(yn))
    assert np.all(np.abs(yn).max(axis=1) > 0)
    # sampled tokens against the per-token oracle
    # every expert's first block, last block and last live row, then random
    # other tokens: 128 in all
    tokens = cover_tokens(d["topk_ids"], cfg.E, 128, 123)
    assert len(tokens) >= 128
    ref, allow = _oracle_tokens(cfg, d, tokens)
    check_close(yn[tokens], ref, BF16_TOL, f"{name} {form} full size, {len(tokens)} tokens", allow)
    # a second run gives bit-identical output (no atomics on the data path)
    assert torch.equal(y_again, y)


def test_fused_experts_on_two_streams_at_once():
    """Two fused_experts calls, each with its own workspace, on two streams
    with no ordering between them: the SM-pair GEMMs take their tile counters
    from each call's workspace, so the calls cannot hand each other's tiles
    out.  The staged entry points on two streams draw different slots of the
    library's counter ring.  Every result equals the single-stream one."""
    cfg = MoEConfig("two", M=1024, H=512, I=512, E=2, topk=2, quant="bf16",
                    routing="softmax", seed=46)
    assert cfg.M * cfg.topk >= 256 * cfg.E            # the SM-pair form
    d = make_inputs(cfg, "cuda")
    y_ref = _run(cfg, d)
    p = moe.Problem.from_config(cfg)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ws = [torch.empty(moe.moe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
          for _ in range(2)]
    ys = [torch.zeros_like(d["x"]) for _ in range(2)]
    bs = [moe.stage_buffers(p) for _ in range(2)]
    torch.cuda.synchronize()
    for _ in range(6):
        for j, s in enumerate((s1, s2)):
            moe.fused_experts(p, d["x"], d["w13"], None, d["w2"], None, d["topk_weights"],
                              d["topk_ids"], ys[j], ws[j], stream=s)
        for j, s in enumerate((s1, s2)):
            b = bs[j]
            moe.moe_align_permute(p, d["x"], d["topk_ids"], None, b["sorted_ids"],
                                  b["block_expert_ids"], b["expert_offsets"],
                                  b["num_post_padded"], b["inv_perm"], b["x_perm"], None,
                                  b["align_ws"], stream=s)
            moe.grouped_gemm_w13(p, b["x_perm"], None, d["w13"], None, b["block_expert_ids"],
                                 b["num_post_padded"], b["z"], None, fuse_act=True, stream=s)
            moe.grouped_gemm_w2(p, b["z"], None, d["w2"], None, b["block_expert_ids"],
                                b["num_post_padded"], b["y2"], stream=s)
            moe.unpermute_reduce(p, b["y2"], b["inv_perm"], d["topk_weights"], b["y"], stream=s)
    torch.cuda.synchronize()
    assert moe.moe_sync_status() == 0
    for j in range(2):
        assert torch.equal(ys[j], y_ref)
        assert torch.equal(bs[j]["y"], y_ref)
