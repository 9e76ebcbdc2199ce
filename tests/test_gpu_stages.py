"""GPU parity of stages 2-5 one at a time (bf16 path): grouped GEMM1 (plain
and with the fused SiLU-and-mul epilogue), SiLU-and-mul, grouped GEMM2 and
the weighted unpermute-reduce, against the fp64 oracle on the same inputs.
Expert loads are ragged (0, 1, 127, 128, 129, ... rows) so tiles are full,
nearly empty and split across blocks."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from oracle import codecs, experts, routing

from .gpu_util import (BF16_TOL, QUANT_TOL, act_allowance, bf16_gemm_form, check_close,
                       flip_allowance, np32)

pytestmark = pytest.mark.gpu


def _ragged_problem(counts, H, I, seed=0, topk=1):
    """topk_ids giving expert e exactly counts[e] routed items (k = 1)."""
    E = len(counts)
    ids = np.concatenate([np.full(c, e, dtype=np.int32) for e, c in enumerate(counts)])
    rng = np.random.default_rng(seed)
    rng.shuffle(ids)
    M = len(ids)
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, H, generator=g).to(torch.bfloat16)
    w13 = (torch.randn(E, 2 * I, H, generator=g) * 0.02).to(torch.bfloat16)
    w2 = (torch.randn(E, H, I, generator=g) * 0.02).to(torch.bfloat16)
    w = torch.rand(M, 1, generator=g)
    return dict(x=x, ids=torch.from_numpy(ids).view(M, 1), w=w, w13=w13, w2=w2, E=E, M=M)


RAGGED = [
    ([0, 1, 127, 128, 129, 300], 256, 256),
    ([5, 0, 0, 260], 512, 384),
    ([128], 256, 128),
]


def _staged(d, H, I, fuse):
    p = moe.Problem(M=d["M"], H=H, I=I, E=d["E"], topk=1)
    b = moe.stage_buffers(p)
    dev = {k: v.cuda() for k, v in d.items() if isinstance(v, torch.Tensor)}
    moe.moe_align_permute(p, dev["x"], dev["ids"], None, b["sorted_ids"], b["block_expert_ids"],
                          b["expert_offsets"], b["num_post_padded"], b["inv_perm"], b["x_perm"],
                          None, b["align_ws"])
    if fuse:
        moe.grouped_gemm_w13(p, b["x_perm"], None, dev["w13"], None, b["block_expert_ids"],
                             b["num_post_padded"], b["z"], None, fuse_act=True)
    else:
        moe.grouped_gemm_w13(p, b["x_perm"], None, dev["w13"], None, b["block_expert_ids"],
                             b["num_post_padded"], b["h1"], None, fuse_act=False)
        moe.act_mul_quant(p, b["h1"], b["num_post_padded"], b["z"], None)
    moe.grouped_gemm_w2(p, b["z"], None, dev["w2"], None, b["block_expert_ids"],
                        b["num_post_padded"], b["y2"])
    moe.unpermute_reduce(p, b["y2"], b["inv_perm"], dev["w"], b["y"])
    assert moe.moe_sync_status() == 0
    return p, b


@pytest.mark.parametrize("counts,H,I", RAGGED)
@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("form", ["single", "pairs"])
def test_stages_bf16_ragged(counts, H, I, fuse, form):
    d = _ragged_problem(counts, H, I)
    with bf16_gemm_form(form):
        p, b = _staged(d, H, I, fuse)
    ids = d["ids"].numpy()
    route = routing.align_permute(ids, d["E"], 128)
    n = route["num_tokens_post_padded"]
    R = d["M"]
    live = route["sorted_token_ids"][:n] < R
    xp, _ = experts.permute_rows(np32(d["x"]), route, 1)
    w13, w2 = np32(d["w13"]), np32(d["w2"])
    h1 = experts.grouped_gemm(xp, None, w13, None, route, 128, "bf16")
    if not fuse:
        check_close(np32(b["h1"])[:n][live], codecs.round_bf16(h1[:n][live]), BF16_TOL, "h1")
        # SiLU-and-mul on the GPU's own h1 (isolates stage 3)
        z_from_gpu_h1 = codecs.round_bf16(experts.act_mul(np32(b["h1"])[:n], I))
        check_close(np32(b["z"])[:n], z_from_gpu_h1, BF16_TOL, "act")
    z = codecs.round_bf16(experts.act_mul(h1, I))
    check_close(np32(b["z"])[:n][live], z[:n][live], BF16_TOL, "z",
                allow=act_allowance(codecs.round_bf16(h1[:n][live]), I))
    # GEMM2 on the GPU's own z (isolates stage 4)
    zg = np.zeros((len(route["sorted_token_ids"]), I))
    zg[:n] = np32(b["z"])[:n]
    y2_iso = experts.grouped_gemm(zg, None, w2, None, route, 128, "bf16")
    check_close(np32(b["y2"])[:n][live], codecs.round_bf16(y2_iso[:n][live]), BF16_TOL, "y2")
    # reduce on the GPU's own y2 (isolates stage 5)
    y2g = np.zeros((len(route["sorted_token_ids"]), H))
    y2g[:n] = np32(b["y2"])[:n]
    y_iso = experts.unpermute_reduce(y2g, route["inv_perm"], np32(d["w"]))
    check_close(np32(b["y"]), y_iso, BF16_TOL, "reduce")
    # whole path
    ref = experts.fused_experts(np32(d["x"]), ids, np32(d["w"]), w13, w2)
    inv = route["inv_perm"]
    items = np.where((inv >= 0)[..., None], ref["y2"][np.maximum(inv, 0)], 0.0)
    check_close(np32(b["y"]), ref["y"], BF16_TOL, "y",
                allow=flip_allowance(ref["y"], items, np32(d["w"])))


SPLIT_CASES = [  # (counts, H, I, topk): ragged loads, top-1 and top-3 with skipped slots
    ([0, 1, 127, 128, 129, 300], 256, 512, 1),
    ([16, 16, 16, 16, 16, 16, 16, 16], 512, 896, 1),
    (None, 512, 640, 3),
]


@pytest.mark.parametrize("counts,H,I,topk", SPLIT_CASES)
def test_gemm2_split_k_stages(counts, H, I, topk):
    """GEMM2 in K slices: each live routed item's slice sums add up to its
    fp32 GEMM2 row (isolated on the GPU's own z), the sliced reduce matches
    the oracle's reduce of the bf16-rounded sums, and both match the unsliced
    stages; every slice count that leaves no slice empty (at most 8) is
    accepted, others are rejected."""
    if counts is None:           # top-3, random experts, a quarter of the slots skipped
        g = torch.Generator().manual_seed(2)
        M, E = 40, 6
        ids = torch.randint(0, E, (M, topk), generator=g, dtype=torch.int32)
        ids[torch.rand(M, topk, generator=g) < 0.25] = -1
        d = _ragged_problem([1] * E, H, I, seed=3)
        d.update(ids=ids, M=M, x=torch.randn(M, H, generator=g).to(torch.bfloat16),
                 w=torch.rand(M, topk, generator=g))
    else:
        d = _ragged_problem(counts, H, I, seed=5)
    p = moe.Problem(M=d["M"], H=H, I=I, E=d["E"], topk=topk)
    b = moe.stage_buffers(p)
    dev = {k: v.cuda() for k, v in d.items() if isinstance(v, torch.Tensor)}
    moe.moe_align_permute(p, dev["x"], dev["ids"], None, b["sorted_ids"], b["block_expert_ids"],
                          b["expert_offsets"], b["num_post_padded"], b["inv_perm"], b["x_perm"],
                          None, b["align_ws"])
    moe.grouped_gemm_w13(p, b["x_perm"], None, dev["w13"], None, b["block_expert_ids"],
                         b["num_post_padded"], b["z"], None, fuse_act=True)
    moe.grouped_gemm_w2(p, b["z"], None, dev["w2"], None, b["block_expert_ids"],
                        b["num_post_padded"], b["y2"])
    moe.unpermute_reduce(p, b["y2"], b["inv_perm"], dev["w"], b["y"])
    assert moe.moe_sync_status() == 0
    ids = d["ids"].numpy()
    route = routing.align_permute(ids, d["E"], 128)
    n = route["num_tokens_post_padded"]
    R = d["M"] * topk
    sid = route["sorted_token_ids"][:n]
    live = sid < R
    zg = np.zeros((len(route["sorted_token_ids"]), I))
    zg[:n] = np32(b["z"])[:n]
    y2_iso = experts.grouped_gemm(zg, None, np32(d["w2"]), None, route, 128, "bf16")
    num_kb = I // 64
    valid = sorted({-(-num_kb // (-(-num_kb // s))) for s in range(1, num_kb + 1)} & set(range(1, 9)))
    assert moe.moe_gemm2_splits(p) in valid or moe.moe_gemm2_splits(p) == 1
    for splits in sorted({1, 2, valid[len(valid) // 2], valid[-1]}):
        part = torch.full((moe.moe_gemm2_partial_bytes(p, splits) // 4,), float("nan"),
                          device="cuda")
        moe.grouped_gemm_w2_split(p, b["z"], dev["w2"], b["block_expert_ids"],
                                  b["num_post_padded"], b["sorted_ids"], splits, part)
        y = torch.empty_like(b["y"])
        moe.unpermute_reduce_split(p, part, splits, b["inv_perm"], dev["w"], y)
        assert moe.moe_sync_status() == 0
        ps = np32(part).reshape(splits, R, H).astype(np.float64).sum(axis=0)
        # slice sums of each live routed item against its GEMM2 row
        check_close(ps[sid[live]], y2_iso[:n][live], BF16_TOL, f"slice sums s={splits}")
        # the sliced reduce = the oracle's reduce of the bf16-rounded slice sums
        y2_pad = np.zeros((len(route["sorted_token_ids"]), H))
        y2_pad[:n][live] = codecs.round_bf16(ps[sid[live]])
        inv = route["inv_perm"]
        y_iso = experts.unpermute_reduce(y2_pad, inv, np32(d["w"]))
        check_close(np32(y), y_iso, BF16_TOL, f"split reduce s={splits}")
        # and the unsliced stages, up to one flip of each stored Y2 row
        items = np.where((inv >= 0)[..., None], np32(b["y2"])[np.maximum(inv, 0)], 0.0)
        check_close(np32(y), np32(b["y"]).astype(np.float64), BF16_TOL,
                    f"split vs unsplit s={splits}",
                    allow=flip_allowance(np32(b["y"]), items, np32(d["w"])))
    bad = [s for s in range(2, num_kb + 2) if s not in valid][:1] + [9]   # at most 8 slices
    for splits in bad:
        part = torch.empty(moe.moe_gemm2_partial_bytes(p, splits) // 4, device="cuda")
        with pytest.raises(moe.MoEError):
            moe.grouped_gemm_w2_split(p, b["z"], dev["w2"], b["block_expert_ids"],
                                      b["num_post_padded"], b["sorted_ids"], splits, part)


def test_act_mul_quant_fp8():
    """Stage 3 with dynamic 1x128 FP8 output on random bf16 h1 rows."""
    I, rows = 512, 384
    p = moe.Problem(M=rows, H=256, I=I, E=1, topk=1, quant="fp8")
    g = torch.Generator().manual_seed(3)
    h1 = (torch.randn(rows, 2 * I, generator=g) * 3).to(torch.bfloat16)
    npp = torch.tensor([rows], dtype=torch.int32)
    for fmt in ("fp32", "ue8m0"):
        p = moe.Problem(M=rows, H=256, I=I, E=1, topk=1, quant="fp8", act_scale_fmt=fmt)
        z = torch.empty(moe.moe_m_sum_bound(p), I, dtype=torch.uint8, device="cuda")
        zs = torch.empty(moe.moe_m_sum_bound(p), I // 128, dtype=torch.float32, device="cuda")
        moe.act_mul_quant(p, h1.cuda(), npp.cuda(), z, zs)
        assert moe.moe_sync_status() == 0
        zr = experts.act_mul(np32(h1), I)
        q, s = experts.quant_act_1x128(zr, fmt)
        sg = np32(zs)[:rows].astype(np.float64)
        # scales: fp32 of amax/448 on both sides; amax may differ in the last fp32 bit
        np.testing.assert_allclose(sg, s, rtol=2 ** -20)
        deq_g = codecs.e4m3_decode(np32(z)[:rows]) * np.repeat(sg, 128, axis=1)
        deq_r = q * np.repeat(s, 128, axis=1)
        check_close(deq_g, deq_r, QUANT_TOL, "z fp8")
        codes_equal = np.mean(np32(z)[:rows] == codecs.e4m3_encode(q))
        assert codes_equal > 0.999, codes_equal


@pytest.mark.parametrize("quant,fmt", [("fp8", "fp32"), ("fp8", "ue8m0"), ("mxfp8", "ue8m0")])
def test_act_quant_keeps_the_sign_of_zero(quant, fmt):
    """z = SiLU(g) * u is exactly -0 where u = +0 and g < 0 (or u = -0 and
    g > 0): its code is the negative zero 0x80, as the IEEE quotient -0 / s
    and the oracle give; +0 gives 0x00."""
    I, rows = 256, 64
    g = torch.Generator().manual_seed(4)
    h1 = (torch.randn(rows, 2 * I, generator=g) * 3).to(torch.bfloat16)
    h1[:, I:I + 32] = 0.0                                    # u = +0
    h1[:, I + 32:I + 64] = -0.0                              # u = -0
    p = moe.Problem(M=rows, H=256, I=I, E=1, topk=1, quant=quant, act_scale_fmt=fmt)
    grp = experts.act_group(quant)
    z = torch.empty(moe.moe_m_sum_bound(p), I, dtype=torch.uint8, device="cuda")
    zs = torch.empty(moe.moe_m_sum_bound(p), I // grp, dtype=torch.float32, device="cuda")
    moe.act_mul_quant(p, h1.cuda(), torch.tensor([rows], dtype=torch.int32).cuda(), z, zs)
    assert moe.moe_sync_status() == 0
    gate = np32(h1)[:, :64]
    want = np.where(np.concatenate([gate[:, :32] < 0, gate[:, 32:] > 0], axis=1), 0x80, 0x00)
    zero_g = gate == 0                                      # SiLU(0) * u = +0 * u
    got = np32(z)[:rows, :64]
    assert np.array_equal(got[~zero_g], want[~zero_g])
    zr = experts.act_mul(np32(h1), I)
    q, _ = experts.quant_act_1x128(zr, fmt, grp)
    assert np.array_equal(codecs.e4m3_encode(q[:, :64]), np.where(zero_g, got, want))


def test_reduce_skips_invalid_slots():
    H, M, k = 1024, 77, 4
    g = torch.Generator().manual_seed(9)
    ids = torch.randint(0, 6, (M, k), generator=g, dtype=torch.int32)
    ids[torch.rand(M, k, generator=g) < 0.3] = -1
    route = routing.align_permute(ids.numpy(), 6, 128)
    cap = len(route["sorted_token_ids"])
    y2 = torch.randn(cap, H, generator=g).to(torch.bfloat16)
    w = torch.rand(M, k, generator=g)
    p = moe.Problem(M=M, H=H, I=128, E=6, topk=k)
    y = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    inv = torch.from_numpy(route["inv_perm"].astype(np.int32))
    moe.unpermute_reduce(p, y2.cuda(), inv.cuda(), w.cuda(), y)
    assert moe.moe_sync_status() == 0
    ref = experts.unpermute_reduce(np32(y2), route["inv_perm"], w.numpy())
    check_close(np32(y), ref, BF16_TOL, "reduce")
