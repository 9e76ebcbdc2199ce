"""Pins for oracle/experts.py.

* the permuted form (the pages' five stages) equals a per-token brute-force
  loop that never permutes;
* E = 1, k = 1, w = 1 reduces the path to a dense SwiGLU MLP, checked against
  torch's fp64 matmul and F.silu;
* the router-weight placement invariant W^T(a z) = a W^T z;
* the FP8 block formula equals dequantise-then-multiply;
* activation quantisation checked against torch's float8 cast and the e4m3
  error bound;
* planted mistakes (in the oracle, on the CPU) are caught by these pins.
"""
import numpy as np
import pytest
import torch

from moe_synth import MoEConfig, make_inputs
from oracle import codecs, experts, routing


def _np(t):
    return None if t is None else (t.float().numpy() if t.dtype in (torch.bfloat16,)
                                   else t.numpy())


def _inputs(cfg):
    d = make_inputs(cfg)
    return dict(x=_np(d["x"]), topk_ids=_np(d["topk_ids"]), topk_weights=_np(d["topk_weights"]),
                w13=_np(d["w13"]), w2=_np(d["w2"]), w13_scale=_np(d["w13_scale"]),
                w2_scale=_np(d["w2_scale"]))


SMALL = {
    "bf16": MoEConfig("t_bf16", M=16, H=256, I=128, E=8, topk=2, quant="bf16",
                      routing="softmax", seed=1),
    "fp8": MoEConfig("t_fp8", M=12, H=256, I=256, E=4, topk=2, quant="fp8",
                     routing="softmax", seed=11),
    "fp8_ue8m0": MoEConfig("t_fp8u", M=12, H=256, I=256, E=4, topk=2, quant="fp8",
                           routing="softmax", seed=12, act_scale_fmt="ue8m0"),
    "mxfp4": MoEConfig("t_mx", M=10, H=256, I=128, E=4, topk=3, quant="mxfp4",
                       routing="uniform", seed=13, act_scale_fmt="ue8m0"),
    "invalid": MoEConfig("t_inv", M=20, H=128, I=128, E=6, topk=3, quant="bf16",
                         routing="softmax", seed=14, invalid_frac=0.3),
    "mxfp8": MoEConfig("t_mx8", M=10, H=256, I=128, E=4, topk=3, quant="mxfp8",
                       routing="uniform", seed=15, act_scale_fmt="ue8m0"),
}


def _both_forms(cfg, exact=False, block_size=128):
    a = _inputs(cfg)
    kw = dict(quant=cfg.quant, act_scale_fmt=cfg.act_scale_fmt,
              apply_router_weight_on_input=cfg.apply_router_weight_on_input, exact=exact)
    f2 = experts.fused_experts(**a, block_size=block_size, **kw)["y"]
    f1 = experts.fused_experts_per_token(**a, **kw)
    return f1, f2


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("exact", [False, True])
def test_permuted_form_equals_per_token_loop(name, exact):
    f1, f2 = _both_forms(SMALL[name], exact=exact)
    assert np.all(np.isfinite(f2))
    rms = np.sqrt(np.mean(f1 ** 2))
    np.testing.assert_allclose(f2, f1, rtol=1e-12, atol=1e-12 * rms)


def test_block_size_does_not_change_result():
    cfg = SMALL["bf16"]
    a = _inputs(cfg)
    ys = [experts.fused_experts(**a, block_size=A)["y"] for A in (16, 32, 64, 128)]
    for y in ys[1:]:
        np.testing.assert_allclose(y, ys[0], rtol=1e-12, atol=0)


def test_dense_special_case_is_swiglu_mlp():
    """E=1, k=1, w=1: y = W2 (silu(Wg x) * (Wu x)) -- a dense SwiGLU MLP."""
    g = torch.Generator().manual_seed(5)
    M, H, I = 7, 128, 256
    x = torch.randn(M, H, generator=g, dtype=torch.float64)
    w13 = torch.randn(1, 2 * I, H, generator=g, dtype=torch.float64) * 0.05
    w2 = torch.randn(1, H, I, generator=g, dtype=torch.float64) * 0.05
    ref = (torch.nn.functional.silu(x @ w13[0, :I].T) * (x @ w13[0, I:].T)) @ w2[0].T
    out = experts.fused_experts(x.numpy(), np.zeros((M, 1), np.int64), np.ones((M, 1)),
                                w13.numpy(), w2.numpy(), exact=True)["y"]
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-14)


def test_router_weight_placement_invariant():
    """Scaling Z rows by w before W2 equals scaling the W2 output (exact mode)."""
    cfg = SMALL["bf16"]
    a = _inputs(cfg)
    E, A, k = a["w13"].shape[0], 128, cfg.topk
    route = routing.align_permute(a["topk_ids"], E, A)
    xp, _ = experts.permute_rows(a["x"], route, k)
    z = experts.act_mul(experts.grouped_gemm(xp, None, a["w13"], None, route, A, "bf16"),
                        cfg.I, exact=True)
    R = cfg.M * k
    sid = route["sorted_token_ids"]
    w_row = np.where(sid < R, a["topk_weights"].reshape(-1)[np.minimum(sid, R - 1)], 0.0)
    y_in = experts.unpermute_reduce(
        experts.grouped_gemm(z * w_row[:, None], None, a["w2"], None, route, A, "bf16"),
        route["inv_perm"], a["topk_weights"], apply_router_weight_on_input=True, exact=True)
    y_out = experts.unpermute_reduce(
        experts.grouped_gemm(z, None, a["w2"], None, route, A, "bf16"),
        route["inv_perm"], a["topk_weights"], exact=True)
    np.testing.assert_allclose(y_in, y_out, rtol=1e-12, atol=1e-15)


def test_apply_router_weight_on_input_topk1():
    cfg = SMALL["bf16"].with_(topk=1, apply_router_weight_on_input=True, seed=21)
    f1, f2 = _both_forms(cfg)
    np.testing.assert_allclose(f2, f1, rtol=1e-12, atol=0)
    # for top-1 it matches output weighting up to bf16 rounding of the scaled input
    a = _inputs(cfg)
    y_out = experts.fused_experts(**a)["y"]
    rms = np.sqrt(np.mean(y_out ** 2))
    assert np.max(np.abs(f2 - y_out)) <= 2e-2 * rms
    with pytest.raises(ValueError):
        experts.fused_experts(**_inputs(SMALL["bf16"]), apply_router_weight_on_input=True)


def test_fp8_block_formula_equals_dequantised_product():
    cfg = SMALL["fp8"]
    a = _inputs(cfg)
    A = 128
    route = routing.align_permute(a["topk_ids"], cfg.E, A)
    xq, xs = experts.permute_rows(a["x"], route, cfg.topk, scale_fmt="fp32")
    c = experts.grouped_gemm(xq, xs, a["w13"], a["w13_scale"], route, A, "fp8")
    wd = experts.dequant_weights(a["w13"], a["w13_scale"], "fp8")
    rows = routing.row_expert_ids(route, A)
    blocks = route["block_expert_ids"]
    ref = np.zeros_like(c)
    for b in range(route["num_tokens_post_padded"] // A):
        sl = slice(b * A, (b + 1) * A)
        ref[sl] = (xq[sl] * np.repeat(xs[sl], 128, axis=1)) @ wd[blocks[b]].T
    np.testing.assert_allclose(c, ref, rtol=1e-12, atol=1e-12)
    assert np.all(c[rows == -1] == 0)


def test_activation_quant_against_torch_cast():
    rng = np.random.default_rng(3)
    v = codecs.round_bf16(rng.normal(0, 1, (64, 512)) * rng.uniform(0.01, 100, (64, 1)))
    q, s = experts.quant_act_1x128(v, "fp32")
    vt = torch.from_numpy(v.astype(np.float32)).view(64, 4, 128)
    st = (vt.abs().amax(-1).clamp_min(float(np.float32(1e-10))) / 448.0)
    qt = (vt / st[..., None]).to(torch.float8_e4m3fn).double().view(64, 512)
    assert np.array_equal(s, st.double().numpy())
    assert np.array_equal(q, qt.numpy())
    # the amax element of each group maps to +-448
    g = np.abs(q.reshape(64, 4, 128)).max(-1)
    assert np.all(g == 448.0)
    # reconstruction within e4m3 half-ulp (2^-4 relative for normal codes)
    rec = q * np.repeat(s, 128, axis=1)
    big = np.abs(v) >= 2.0 ** -6 * np.repeat(s, 128, axis=1)
    assert np.all(np.abs(rec - v)[big] <= 2.0 ** -4 * np.abs(v)[big] * (1 + 1e-6))


def test_activation_quant_ue8m0_and_zero_group():
    rng = np.random.default_rng(4)
    v = codecs.round_bf16(rng.normal(0, 3, (8, 256)))
    v[0, :128] = 0.0
    q32, s32 = experts.quant_act_1x128(v, "fp32")
    q8, s8 = experts.quant_act_1x128(v, "ue8m0")
    assert np.all(codecs.ceil_pow2(s8) == s8) and np.all(s8 >= s32) and np.all(s8 < 2 * s32)
    assert np.all(q8[0, :128] == 0) and s32[0, 0] == codecs.round_fp32(np.float32(1e-10) / 448.0)
    assert np.all(np.abs(q8) <= 448.0)


def test_invalid_ids_contribute_nothing():
    cfg = SMALL["invalid"]
    a = _inputs(cfg)
    assert np.any(a["topk_ids"] < 0)
    y = experts.fused_experts(**a)["y"]
    w2 = a["topk_weights"].copy()
    w2[a["topk_ids"] < 0] = 123.0
    a2 = dict(a, topk_weights=w2)
    assert np.array_equal(experts.fused_experts(**a2)["y"], y)


def test_empty_batch():
    cfg = SMALL["bf16"]
    a = _inputs(cfg)
    a = dict(a, x=a["x"][:0], topk_ids=a["topk_ids"][:0], topk_weights=a["topk_weights"][:0])
    assert experts.fused_experts(**a)["y"].shape == (0, cfg.H)


def test_silu_against_scipy_and_identity():
    from scipy.special import expit
    g = np.linspace(-30, 30, 2001)
    np.testing.assert_allclose(experts.silu(g), g * expit(g), rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(experts.silu(-g), experts.silu(g) - g, rtol=1e-12, atol=1e-12)
    assert experts.silu(0.0) == 0.0


# --------------------------------------------------------------- planted mistakes
def _catches(monkeypatch, target, replacement):
    """Plant ``replacement`` for ``target`` in the oracle and report whether a
    pin now fails."""
    monkeypatch.setattr(experts, target, replacement)
    failures = 0
    for fn in (lambda: test_dense_special_case_is_swiglu_mlp(),
               lambda: test_permuted_form_equals_per_token_loop("bf16", False),
               lambda: test_permuted_form_equals_per_token_loop("fp8", False)):
        try:
            fn()
        except AssertionError:
            failures += 1
    return failures > 0


def test_planted_gate_up_swap_is_caught(monkeypatch):
    orig = experts.act_mul

    def swapped(h1, I, exact=False, recipe=None):
        h1 = np.asarray(h1)
        return orig(np.concatenate([h1[:, I:], h1[:, :I]], axis=1), I, exact, recipe)
    assert _catches(monkeypatch, "act_mul", swapped)


def test_planted_token_index_mistake_is_caught(monkeypatch):
    orig = experts.permute_rows

    def wrong(x, route, topk, topk_weights=None, scale_fmt=None, group=128):
        r2 = dict(route)
        sid = route["sorted_token_ids"].copy()
        R = route["inv_perm"].size
        live = sid < R
        sid[live] = (sid[live] % topk) * topk + (sid[live] // topk) % topk  # r % k for r // k
        r2["sorted_token_ids"] = sid
        return orig(x, r2, topk, topk_weights, scale_fmt, group)
    assert _catches(monkeypatch, "permute_rows", wrong)


def test_planted_dropped_router_weight_is_caught(monkeypatch):
    orig = experts.unpermute_reduce

    def dropped(y2, inv_perm, topk_weights, apply_router_weight_on_input=False, exact=False):
        return orig(y2, inv_perm, topk_weights, True, exact)
    assert _catches(monkeypatch, "unpermute_reduce", dropped)


def test_planted_fp8_scale_mistake_is_caught(monkeypatch):
    orig = experts.quant_act_1x128

    def wrong(v, scale_fmt="fp32"):
        q, s = orig(v, scale_fmt)
        return q, s * 1.5
    # both forms share the quantiser, so the torch-cast pin is the one that catches it
    monkeypatch.setattr(experts, "quant_act_1x128", wrong)
    with pytest.raises(AssertionError):
        test_activation_quant_against_torch_cast()


@pytest.mark.parametrize("name", ["bf16", "fp8", "mxfp4"])
def test_batched_layout_equals_permuted_form(name):
    """The batched layout's rows through the permuted form (form 2) with one
    slot of weight 1 routed to each row's expert give the same values; rows
    past a count are NaN; counts are clamped to [0, T]."""
    cfg = SMALL[name]
    a = _inputs(cfg)
    E, H, T = cfg.E, cfg.H, 5
    rng = np.random.default_rng(2)
    x_b = np.stack([a["x"][rng.integers(0, cfg.M, T)] for _ in range(E)])     # [E, T, H]
    counts = np.array([T, 0, 3, 9][:E] + [1] * max(0, E - 4))                  # 9 > T: clamped
    kw = dict(quant=cfg.quant, act_scale_fmt=cfg.act_scale_fmt)
    y_b = experts.batched_experts(x_b, counts, a["w13"], a["w2"], a["w13_scale"], a["w2_scale"],
                                  **kw)
    rows, ids = [], []
    for e in range(E):
        c = min(max(int(counts[e]), 0), T)
        rows += [x_b[e, r] for r in range(c)]
        ids += [e] * c
        assert np.all(np.isnan(y_b[e, c:]))
    f2 = experts.fused_experts(np.array(rows), np.array(ids)[:, None], np.ones((len(ids), 1)),
                               a["w13"], a["w2"], a["w13_scale"], a["w2_scale"], **kw)["y"]
    got = np.concatenate([y_b[e, :min(int(counts[e]), T)] for e in range(E)])
    np.testing.assert_array_equal(got, f2)


# ---------------------------------------------------------------- epilogue variants
RECIPE = (1.702, 1.0, 7.0)     # a swigluoai-style setting of the gemm1 recipe


def test_recipe_identity_is_silu_and_clamp_closed_forms():
    rng = np.random.default_rng(9)
    g, u = rng.normal(size=(50, 16)) * 3, rng.normal(size=(50, 16)) * 3
    np.testing.assert_allclose(experts.gated(g, u, (1.0, 0.0, 0.0)), experts.gated(g, u),
                               rtol=1e-15, atol=0)
    # closed forms: g = 0 gives 0; a clamped gate and up; beta shifts the up half
    assert experts.gated(0.0, 5.0, RECIPE) == 0.0
    v = experts.gated(100.0, -50.0, RECIPE)              # g' = 7, u' = -7
    np.testing.assert_allclose(v, (-7.0 + 1.0) * 7.0 / (1.0 + np.exp(-1.702 * 7.0)), rtol=1e-15)
    v = experts.gated(-3.0, 2.0, (2.0, 0.5, 0.0))        # no clamp
    np.testing.assert_allclose(v, 2.5 * -3.0 * special_expit(2.0 * -3.0), rtol=1e-15)


def special_expit(x):
    from scipy import special
    return special.expit(x)


@pytest.mark.parametrize("name", ["bf16", "fp8", "mxfp4"])
def test_router_weight_placement_in_gemm2_is_exact_by_linearity(name):
    """exact mode: scaling GEMM2's rows by the router weight and summing gives
    the default path's result (W2^T (a z) + a b = a (W2^T z + b)); both forms."""
    cfg = SMALL[name]
    a = _inputs(cfg)
    kw = dict(quant=cfg.quant, act_scale_fmt=cfg.act_scale_fmt, exact=True)
    rng = np.random.default_rng(4)
    b2 = rng.normal(size=(cfg.E, cfg.H)) * 0.1
    ref = experts.fused_experts(**a, w2_bias=b2, **kw)["y"]
    f2 = experts.fused_experts(**a, w2_bias=b2, router_weight_in_gemm2=True, **kw)["y"]
    f1 = experts.fused_experts_per_token(**a, w2_bias=b2, router_weight_in_gemm2=True, **kw)
    np.testing.assert_allclose(f2, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(f1, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("name", ["bf16", "fp8", "mxfp4"])
def test_epilogue_variants_both_forms_agree(name):
    cfg = SMALL[name]
    a = _inputs(cfg)
    rng = np.random.default_rng(5)
    kw = dict(quant=cfg.quant, act_scale_fmt=cfg.act_scale_fmt,
              w13_bias=codecs.round_bf16(rng.normal(size=(cfg.E, 2 * cfg.I)) * 0.5),
              w2_bias=codecs.round_bf16(rng.normal(size=(cfg.E, cfg.H)) * 0.5),
              router_weight_in_gemm2=True, act_recipe=RECIPE)
    f2 = experts.fused_experts(**a, **kw)["y"]
    f1 = experts.fused_experts_per_token(**a, **kw)
    np.testing.assert_allclose(f1, f2, rtol=0, atol=1e-12 * np.sqrt(np.mean(f2 ** 2)))


def test_biases_with_zero_weights_closed_form():
    """W = 0: H1 = b13, so z = gated(b13 gate, b13 up) and y = sum_i w_i b2[e_i]."""
    cfg = SMALL["bf16"]
    a = _inputs(cfg)
    a["w13"] = np.zeros_like(a["w13"])
    a["w2"] = np.zeros_like(a["w2"])
    rng = np.random.default_rng(6)
    b13 = codecs.round_bf16(rng.normal(size=(cfg.E, 2 * cfg.I)))
    b2 = codecs.round_bf16(rng.normal(size=(cfg.E, cfg.H)))
    out = experts.fused_experts(**a, w13_bias=b13, w2_bias=b2, act_recipe=RECIPE)
    ids, w = a["topk_ids"], a["topk_weights"]
    want = np.zeros((cfg.M, cfg.H))
    for t in range(cfg.M):
        for i in range(cfg.topk):
            want[t] += w[t, i] * b2[ids[t, i]]
    np.testing.assert_allclose(out["y"], codecs.round_bf16(want), rtol=0, atol=0)
    zb = codecs.round_bf16(experts.gated(b13[:, :cfg.I], b13[:, cfg.I:], RECIPE))
    e0 = out["route"]["block_expert_ids"][0]
    np.testing.assert_array_equal(out["z"][0], zb[e0])


def test_dense_special_case_with_bias_and_recipe():
    """E=1, k=1, w=1, exact: a dense gated MLP with biases, against torch."""
    g = torch.Generator().manual_seed(8)
    M, H, I = 6, 128, 128
    x = torch.randn(M, H, generator=g, dtype=torch.float64)
    w13 = torch.randn(1, 2 * I, H, generator=g, dtype=torch.float64) * 0.1
    w2 = torch.randn(1, H, I, generator=g, dtype=torch.float64) * 0.1
    b13 = torch.randn(1, 2 * I, generator=g, dtype=torch.float64)
    b2 = torch.randn(1, H, generator=g, dtype=torch.float64)
    h = x @ w13[0].T + b13[0]
    gt, up = h[:, :I].clamp(max=7.0), h[:, I:].clamp(-7.0, 7.0)
    z = (up + 1.0) * gt * torch.sigmoid(1.702 * gt)
    ref = z @ w2[0].T + b2[0]
    out = experts.fused_experts(x.numpy(), np.zeros((M, 1), np.int64), np.ones((M, 1)),
                                w13.numpy(), w2.numpy(), exact=True, w13_bias=b13.numpy(),
                                w2_bias=b2.numpy(), act_recipe=RECIPE)["y"]
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- MXFP8 (1x32)
def test_mxfp8_activation_quant_against_torch_cast():
    """1x32 groups with UE8M0 scales: scale 2^ceil(log2(amax/448)), codes by
    torch's float8 cast."""
    rng = np.random.default_rng(11)
    v = codecs.round_bf16(rng.normal(0, 1, (32, 256)) * rng.uniform(0.01, 100, (32, 1)))
    q, s = experts.quant_act_1x128(v, "ue8m0", 32)
    vt = torch.from_numpy(v.astype(np.float32)).view(32, 8, 32).double()
    st = torch.exp2(torch.ceil(torch.log2(vt.abs().amax(-1) / 448.0)))
    qt = (vt / st[..., None]).float().to(torch.float8_e4m3fn).double().view(32, 256)
    assert np.array_equal(s, st.numpy())
    assert np.array_equal(q, qt.numpy())
    assert np.all(np.abs(q) <= 448.0) and s.shape == (32, 8)


def test_mxfp8_weight_dequant_against_torch():
    rng = np.random.default_rng(12)
    codes = rng.integers(0, 256, (2, 8, 64), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0          # the two NaN codes of e4m3fn are never stored
    sc = rng.integers(120, 135, (2, 8, 2), dtype=np.uint8)
    want = (torch.from_numpy(codes).view(torch.float8_e4m3fn).double() *
            torch.exp2(torch.from_numpy(sc.astype(np.float64) - 127.0)).repeat_interleave(32, -1))
    assert np.array_equal(experts.dequant_weights(codes, sc, "mxfp8"), want.numpy())


def test_mxfp8_gemm_is_the_dequantised_product():
    cfg = SMALL["mxfp8"]
    a = _inputs(cfg)
    out = experts.fused_experts(**a, quant="mxfp8", act_scale_fmt="ue8m0", exact=True)
    route = out["route"]
    h1 = experts.grouped_gemm(out["x_perm"], out["x_scale"], a["w13"], a["w13_scale"], route, 128,
                              "mxfp8")
    wd = experts.dequant_weights(a["w13"], a["w13_scale"], "mxfp8")
    xd = out["x_perm"] * np.repeat(out["x_scale"], 32, axis=1)
    ids = route["block_expert_ids"]
    for b in range(route["num_tokens_post_padded"] // 128):
        r = slice(b * 128, b * 128 + 128)
        np.testing.assert_allclose(h1[r], xd[r] @ torch.from_numpy(wd[ids[b]]).numpy().T,
                                   rtol=1e-13, atol=1e-13)


def test_mxfp8_needs_ue8m0_activation_scales():
    cfg = SMALL["mxfp8"]
    a = _inputs(cfg)
    with pytest.raises(ValueError):
        experts.fused_experts(**a, quant="mxfp8", act_scale_fmt="fp32")
