"""GPU parity of fused_experts_batched (the BatchedExperts layout [E, T, H]
with per-expert counts) against the oracle: ragged counts (0, 1, a partial
block, a full buffer, a count past T that is clamped), both bf16 tile forms,
FP8 and MXFP4, the decode shape, and a CUDA-graph replay that sees counts
changed on the device after capture."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import CONFIGS, MoEConfig, make_inputs
from oracle import experts

from .gpu_util import BF16_TOL, QUANT_TOL, bf16_gemm_form, check_close, flip_allowance, np32

pytestmark = pytest.mark.gpu


def _case(cfg, T, counts, seed):
    d = make_inputs(cfg, "cuda")
    g = torch.Generator().manual_seed(seed)
    x_b = torch.randn(cfg.E, T, cfg.H, generator=g).to(torch.bfloat16).cuda()
    cnt = torch.tensor(counts, dtype=torch.int32, device="cuda")
    return d, x_b, cnt


def _run(cfg, d, x_b, cnt, expected_m=0, y=None, ws=None):
    p = moe.Problem.from_config(cfg)
    T = x_b.shape[1]
    if ws is None:
        ws = torch.empty(moe.moe_batched_workspace_bytes(p, T), dtype=torch.uint8, device="cuda")
    if y is None:
        y = torch.zeros_like(x_b)
    moe.fused_experts_batched(p, x_b, cnt, d["w13"], d["w13_scale"], d["w2"], d["w2_scale"], y,
                              ws, expected_m=expected_m)
    return y


def _check(cfg, d, x_b, counts, y, tol, rows=None):
    E, T, H = x_b.shape
    ref = experts.batched_experts(np32(x_b), counts, np32(d["w13"]), np32(d["w2"]),
                                  np32(d.get("w13_scale")), np32(d.get("w2_scale")),
                                  quant=cfg.quant, act_scale_fmt=cfg.act_scale_fmt)
    yn = np32(y)
    for e in range(E):
        c = min(max(int(counts[e]), 0), T)
        sel = list(range(c)) if rows is None else [r for r in rows if r < c]
        if not sel:
            continue
        r_ref, r_got = ref[e, sel], yn[e, sel]
        check_close(r_got, r_ref, tol, f"expert {e}",
                    flip_allowance(r_ref, r_ref[:, None, :], np.ones((len(sel), 1))))


BF16 = MoEConfig("bt", M=1, H=512, I=256, E=5, topk=1, quant="bf16", routing="softmax", seed=71)
COUNTS = [0, 1, 130, 256, 300]          # 300 > T: clamped to 256


@pytest.mark.parametrize("form,expected_m", [("auto", 0), ("auto", 300), ("single", 0),
                                             ("pairs", 0)])
def test_batched_bf16_ragged_counts(form, expected_m):
    d, x_b, cnt = _case(BF16, 256, COUNTS, 1)
    with bf16_gemm_form(form):
        y = _run(BF16, d, x_b, cnt, expected_m)
    assert moe.moe_sync_status() == 0
    _check(BF16, d, x_b, COUNTS, y, BF16_TOL)


@pytest.mark.parametrize("quant,fmt", [("fp8", "fp32"), ("fp8", "ue8m0"), ("mxfp4", "ue8m0")])
def test_batched_quantised(quant, fmt):
    """Bit-exact with the standard path on the same rows (one slot of weight
    1 per row: same kernels, same per-row quantisation); against the oracle
    where the activation scales are powers of two.  With fp32 1x128 scales a
    one-ulp difference in H1 (accumulation order) can move a z group's scale
    and re-round all its codes, so that comparison is made stage by stage on
    the GPU's own intermediates (test_gpu_fp8)."""
    cfg = MoEConfig("bq", M=1, H=512, I=256, E=4, topk=1, quant=quant, routing="uniform",
                    seed=72, act_scale_fmt=fmt)
    counts = [3, 0, 256, 129]
    d, x_b, cnt = _case(cfg, 256, counts, 2)
    y = _run(cfg, d, x_b, cnt)
    assert moe.moe_sync_status() == 0
    rows = torch.cat([x_b[e, :c] for e, c in enumerate(counts)])
    ids = torch.cat([torch.full((c, 1), e, dtype=torch.int32) for e, c in enumerate(counts)])
    M = rows.shape[0]
    p2 = moe.Problem.from_config(cfg.with_(M=M))
    ws = torch.empty(moe.moe_workspace_bytes(p2), dtype=torch.uint8, device="cuda")
    y_std = torch.empty_like(rows)
    moe.fused_experts(p2, rows, d["w13"], d["w13_scale"], d["w2"], d["w2_scale"],
                      torch.ones(M, 1, device="cuda"), ids.cuda(), y_std, ws)
    assert moe.moe_sync_status() == 0
    assert torch.equal(torch.cat([y[e, :c] for e, c in enumerate(counts)]), y_std)
    if fmt == "ue8m0":
        _check(cfg, d, x_b, counts, y, QUANT_TOL)


def test_batched_decode_shape_sampled():
    """Mixtral-shaped decode: E = 8, H = 4096, I = 14336, 128-row buffers
    holding the decode routing's ~16 tokens per expert."""
    cfg = CONFIGS["decode"]
    counts = np.bincount(make_inputs(cfg, "cpu", weights=False)["topk_ids"].numpy().ravel(),
                         minlength=cfg.E).tolist()
    d, x_b, cnt = _case(cfg, 128, counts, 3)
    y = _run(cfg, d, x_b, cnt, expected_m=16)
    assert moe.moe_sync_status() == 0
    _check(cfg, d, x_b, counts, y, BF16_TOL, rows=[0, 3, 7, 15, 20])


def test_batched_graph_replay_sees_new_counts():
    d, x_b, cnt = _case(BF16, 256, COUNTS, 4)
    p = moe.Problem.from_config(BF16)
    ws = torch.empty(moe.moe_batched_workspace_bytes(p, 256), dtype=torch.uint8, device="cuda")
    y = torch.zeros_like(x_b)
    _run(BF16, d, x_b, cnt, y=y, ws=ws)               # first call outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _run(BF16, d, x_b, cnt, y=y, ws=ws)
    new_counts = [256, 17, 0, 128, 5]
    cnt.copy_(torch.tensor(new_counts, dtype=torch.int32))
    y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert moe.moe_sync_status() == 0
    direct = _run(BF16, d, x_b, cnt)
    for e, c in enumerate(new_counts):
        assert torch.equal(y[e, :c], direct[e, :c])
    _check(BF16, d, x_b, new_counts, y, BF16_TOL)


def test_batched_rejects_bad_sizes():
    d, x_b, cnt = _case(BF16, 256, COUNTS, 5)
    p = moe.Problem.from_config(BF16)
    assert moe.moe_batched_workspace_bytes(p, 100) == 0     # not a multiple of 128
    with pytest.raises(moe.MoEError) as ei:
        _run(BF16, d, x_b[:, :192].contiguous(), cnt)
    assert ei.value.status == 1
