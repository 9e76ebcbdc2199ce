"""Expert computation of the fused MoE forward -- fp64 oracle.

Test infrastructure only.  Sources (page titles and sections):

* "fused_moe.py 分析" §1.1-1.4: y_t = sum_i alpha_{t,i} f_{e_{t,i}}(x_t); routed
  form C[r, n] = sum_k A[t(r), k] B[e(r), n, k] (B stored [E, N, K]); the
  router-weight placement equivalence W^T(a z) = a W^T z.
* same page, "fused_moe_kernel 的核心原理": fp32 accumulation, cast to the
  compute type; "FP8 W8A8": block-wise C_block ~ dot(qA, qB) * a_scale * b_scale
  per K block.
* "Blackwell 上的 DeepGEMM FusedMoE（vLLM）" §1.1 / §2.6: permute -> GEMM1 (bf16
  mm1_out [M_sum, 2I]) -> SwiGLU + dynamic 1x128 quant -> GEMM2 (bf16 mm2_out)
  -> ep_gather (fp32 weighted sum in slot order, cast to bf16); padding rows
  carry zero activation scales; ids < 0 contribute nothing; with
  apply_router_weight_on_input the reduce uses all-ones weights.

Readings (the pages are silent or disagree):
* gated activation: z = SiLU(first half) * second half of GEMM1's 2I outputs
  (SwiGLU; "SiLU-and-mul"), SiLU(g) = g / (1 + exp(-g));
* intermediate roundings: H1, Z (bf16 mode) and Y2 are rounded to bf16, the
  final y to bf16; everything else is fp64.  ``exact=True`` skips them;
* FP8 activation quant per 1x128 group: s = fp32(max(amax, eps) / 448) with
  eps = fp32(1e-10); UE8M0 option: s rounded up to a power of two; code =
  e4m3_rne_sat(fp32(v / s)).  Padding rows: codes 0, scale 0;
* apply_router_weight_on_input (top-k = 1 only): the routed row is
  bf16(fp32(x_t * w)) before quantisation, and the reduce uses weight 1;
* MXFP4 weights are dequantised (E2M1 * 2^(e-127)) and multiplied in fp64,
  which equals the per-32 block-scaled product exactly.
"""
from __future__ import annotations

import numpy as np

from . import codecs
from .routing import align_permute

EPS32 = float(np.float32(1e-10))


# ----------------------------------------------------------------- quantisation
def quant_act_1x128(v, scale_fmt: str = "fp32", group: int = 128):
    """Dynamic per-(row, column group) FP8 quantisation, groups of 128 (the
    FP8 block and W4A8 recipes) or 32 (MXFP8, always with UE8M0 scales).

    v: [R, K] fp64 (K % group == 0).  Returns (q values [R, K] fp64 on the
    e4m3 grid, s [R, K/group] fp64 holding fp32 (or power-of-two) scales)."""
    v = np.asarray(v, dtype=np.float64)
    R, K = v.shape
    g = v.reshape(R, K // group, group)
    amax = np.abs(g).max(axis=-1) if R else np.zeros((0, K // group))
    s = codecs.round_fp32(np.maximum(amax, EPS32) / codecs.E4M3_MAX)
    if scale_fmt == "ue8m0":
        s = codecs.ceil_pow2(s)
    elif scale_fmt != "fp32":
        raise ValueError(scale_fmt)
    q = codecs.round_e4m3(codecs.round_fp32(g / s[..., None]))
    return q.reshape(R, K), s


def dequant_weights(w, w_scale, quant: str):
    """Weights in storage format -> fp64 values [E, N, K].

    bf16: values as given.  fp8: e4m3 codes * fp32 128x128 block scale.
    mxfp4: E2M1 codes (packed, low nibble even k) * E8M0 scale per 32 along K.
    mxfp8: e4m3 codes * E8M0 scale per 32 along K.
    """
    if quant == "bf16":
        return np.asarray(w, dtype=np.float64)
    if quant == "fp8":
        q = codecs.e4m3_decode(w)
        s = np.asarray(w_scale, dtype=np.float64)
        s_full = np.repeat(np.repeat(s, 128, axis=1), 128, axis=2)
        return q * s_full[:, : q.shape[1], : q.shape[2]]
    if quant == "mxfp4":
        E, N, Kh = np.asarray(w).shape
        q = codecs.e2m1_decode(codecs.unpack_fp4(w, 2 * Kh))
        s = codecs.e8m0_decode(w_scale)
        return q * np.repeat(s, 32, axis=2)
    if quant == "mxfp8":
        q = codecs.e4m3_decode(w)
        return q * np.repeat(codecs.e8m0_decode(w_scale), 32, axis=2)
    raise ValueError(quant)


def act_group(quant: str) -> int:
    """Activation quantisation group along K: 32 for MXFP8 (recipe (1, 32)),
    else 128."""
    return 32 if quant == "mxfp8" else 128


# ------------------------------------------------------------------ the stages
def permute_rows(x, route, topk: int, topk_weights=None, scale_fmt=None, group: int = 128):
    """Data half of the permute: x_perm[row] = x[sorted_token_ids[row] // k].

    Padding rows are zero.  With ``topk_weights`` (apply_router_weight_on_input)
    the row is bf16(fp32(x_t * w_r)).  With ``scale_fmt`` the rows are
    quantised per 1x128 group; padding rows get code 0 and scale 0.
    Returns (x_perm [cap, H], scale [cap, H/128] or None)."""
    x = np.asarray(x, dtype=np.float64)
    H = x.shape[1]
    sid = route["sorted_token_ids"]
    R = route["inv_perm"].size
    cap = len(sid)
    live = sid < R
    xp = np.zeros((cap, H))
    xp[live] = x[sid[live] // topk]
    if topk_weights is not None:
        w = np.asarray(topk_weights, dtype=np.float64).reshape(-1)
        xp[live] = codecs.round_bf16(codecs.round_fp32(xp[live] * w[sid[live]][:, None]))
    if scale_fmt is None:
        return xp, None
    q, s = quant_act_1x128(xp, scale_fmt, group)
    q[~live] = 0.0
    s[~live] = 0.0
    return q, s


def grouped_gemm(a, a_scale, w, w_scale, route, block_size: int, quant: str):
    """C[row, n] = sum_k A[row, k] * W[e, n, k] for every padded block with
    expert e >= 0 below num_tokens_post_padded; other rows are 0.

    bf16: plain fp64 product.  fp8 (block 128x128 weight scales, 1x128
    activation scales): C = sum_kb sa[row, kb] * sb[e, n/128, kb] *
    sum_{k in kb} qa * qb.  mxfp4: A = qa * sa (per 128), W dequantised.
    mxfp8: A = qa * sa (per 32), W dequantised (E8M0 per 32).
    Returns fp64 [cap, N] (not rounded)."""
    a = np.asarray(a, dtype=np.float64)
    cap, K = a.shape
    block_ids = route["block_expert_ids"]
    n_blocks = route["num_tokens_post_padded"] // block_size
    E = np.asarray(w).shape[0]
    if quant == "fp8":
        N = np.asarray(w).shape[1]
    elif quant == "mxfp4":
        N = np.asarray(w).shape[1]
    else:
        N = np.asarray(w).shape[1]
    out = np.zeros((cap, N))
    for b in range(n_blocks):
        e = int(block_ids[b])
        if e < 0:
            continue
        rows = slice(b * block_size, (b + 1) * block_size)
        if quant == "bf16":
            out[rows] = a[rows] @ np.asarray(w[e], dtype=np.float64).T
        elif quant == "fp8":
            qb = codecs.e4m3_decode(w[e])                  # [N, K]
            sb = np.asarray(w_scale[e], dtype=np.float64)  # [N/128, K/128]
            acc = np.zeros((block_size, N))
            for kb in range(K // 128):
                ks = slice(kb * 128, (kb + 1) * 128)
                part = a[rows, ks] @ qb[:, ks].T            # exact: e4m3 products
                sb_n = np.repeat(sb[:, kb], 128)[:N]
                acc += a_scale[rows, kb][:, None] * sb_n[None, :] * part
            out[rows] = acc
        elif quant in ("mxfp4", "mxfp8"):
            wd = dequant_weights(np.asarray(w[e])[None], np.asarray(w_scale[e])[None], quant)[0]
            ad = a[rows] * np.repeat(a_scale[rows], act_group(quant), axis=1)
            out[rows] = ad @ wd.T
        else:
            raise ValueError(quant)
    return out


def silu(g):
    """SiLU(g) = g * sigmoid(g) = g / (1 + exp(-g))."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def gated(g, u, recipe=None):
    """The gated activation of GEMM1's gate and up halves.  recipe None:
    SiLU(g) * u.  recipe (alpha, beta, limit) -- the gemm1_alpha / gemm1_beta /
    gemm1_clamp_limit recipe (page "Blackwell 上的 DeepGEMM FusedMoE（vLLM）",
    §2.6.4; alpha = 1, beta = 0 is SiLU-and-mul): with limit > 0 the gate is
    clamped from above and the up half to [-limit, limit], then
    z = (u + beta) * g * sigmoid(alpha * g)."""
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    if recipe is None:
        return silu(g) * u
    alpha, beta, limit = (float(v) for v in recipe)
    if limit > 0:
        g = np.minimum(g, limit)
        u = np.clip(u, -limit, limit)
    return (u + beta) * g / (1.0 + np.exp(-alpha * g))


def act_mul(h1, I: int, exact: bool = False, recipe=None):
    """SiLU-and-mul on the 2I outputs of GEMM1: z = SiLU(h[:, :I]) * h[:, I:]
    (or the gated recipe).  Unless ``exact``, h1 is first rounded to bf16
    (mm1_out is bf16)."""
    h1 = np.asarray(h1, dtype=np.float64)
    if not exact:
        h1 = codecs.round_bf16(h1)
    return gated(h1[:, :I], h1[:, I:], recipe)


def add_expert_bias(c, bias, route, block_size: int):
    """c[row] += bias[e] for the rows of every used block of expert e (the
    GEMM epilogue's bias, page "fused_moe.py 分析", fused_moe_kernel
    post-processing: dequant -> bias -> router weight -> cast)."""
    if bias is None:
        return c
    c = np.array(c, dtype=np.float64)
    bias = np.asarray(bias, dtype=np.float64)
    ids = route["block_expert_ids"]
    for b in range(route["num_tokens_post_padded"] // block_size):
        if ids[b] >= 0:
            c[b * block_size:(b + 1) * block_size] += bias[ids[b]]
    return c


def unpermute_reduce(y2, inv_perm, topk_weights, apply_router_weight_on_input=False,
                     exact: bool = False):
    """y[t] = sum_{i: inv_perm[t,i] >= 0} w'[t,i] * Y2[inv_perm[t,i]], slot order,
    w' = 1 with apply_router_weight_on_input; cast to bf16 unless ``exact``."""
    y2 = np.asarray(y2, dtype=np.float64)
    inv = np.asarray(inv_perm, dtype=np.int64)
    w = np.asarray(topk_weights, dtype=np.float64)
    M, k = inv.shape
    y = np.zeros((M, y2.shape[1]))
    for i in range(k):
        ok = inv[:, i] >= 0
        wi = np.ones(M) if apply_router_weight_on_input else w[:, i]
        y[ok] += wi[ok, None] * y2[inv[ok, i]]
    return y if exact else codecs.round_bf16(y)


# ------------------------------------------------------------- whole forward
def _act_scale_fmt(quant: str, act_scale_fmt: str):
    if quant == "mxfp8" and act_scale_fmt != "ue8m0":
        raise ValueError("MXFP8 activations take UE8M0 scales")
    return None if quant == "bf16" else act_scale_fmt


def fused_experts(x, topk_ids, topk_weights, w13, w2, w13_scale=None, w2_scale=None, *,
                  quant="bf16", act_scale_fmt="fp32", block_size=128,
                  apply_router_weight_on_input=False, exact=False, w13_bias=None,
                  w2_bias=None, router_weight_in_gemm2=False, act_recipe=None):
    """Form 2 (the pages' organisation): routing, permute, grouped GEMM1,
    SiLU-and-mul (+ quant), grouped GEMM2, weighted unpermute-reduce.
    Epilogue variants: expert biases added to the GEMM sums before rounding,
    the router weight applied to GEMM2's rows before their rounding (the
    reduce then only sums), the gated activation recipe (see ``gated``).
    Returns a dict with every intermediate and ``y`` [M, H]."""
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(topk_ids)
    M, k = ids.shape
    E = np.asarray(w13).shape[0]
    I = np.asarray(w2).shape[2] if quant != "mxfp4" else 2 * np.asarray(w2).shape[2]
    if apply_router_weight_on_input and k != 1:
        raise ValueError("apply_router_weight_on_input needs top-k = 1")
    if apply_router_weight_on_input and router_weight_in_gemm2:
        raise ValueError("the router weight is applied once")
    fmt = _act_scale_fmt(quant, act_scale_fmt)
    route = align_permute(ids, E, block_size)
    xp, xs = permute_rows(x, route, k,
                          topk_weights if apply_router_weight_on_input else None, fmt,
                          act_group(quant))
    h1 = grouped_gemm(xp, xs, w13, w13_scale, route, block_size, quant)
    h1 = add_expert_bias(h1, w13_bias, route, block_size)
    z = act_mul(h1, I, exact=exact, recipe=act_recipe)
    if fmt is None:
        zq, zs = (z if exact else codecs.round_bf16(z)), None
    else:
        zq, zs = quant_act_1x128(z, fmt, act_group(quant))
        live = route["sorted_token_ids"] < M * k
        zq[~live] = 0.0
        zs[~live] = 0.0
    y2 = grouped_gemm(zq, zs, w2, w2_scale, route, block_size, quant)
    y2 = add_expert_bias(y2, w2_bias, route, block_size)
    if router_weight_in_gemm2:
        sid = route["sorted_token_ids"]
        wflat = np.asarray(topk_weights, dtype=np.float64).reshape(-1)
        row_w = np.where(sid < M * k, wflat[np.minimum(sid, M * k - 1)], 0.0)
        y2 = y2 * row_w[:, None]
    if not exact:
        y2 = codecs.round_bf16(y2)
    y = unpermute_reduce(y2, route["inv_perm"], topk_weights,
                         apply_router_weight_on_input or router_weight_in_gemm2, exact=exact)
    return {"route": route, "x_perm": xp, "x_scale": xs, "h1": h1, "z": zq, "z_scale": zs,
            "y2": y2, "y": y}


def fused_experts_per_token(x, topk_ids, topk_weights, w13, w2, w13_scale=None,
                            w2_scale=None, *, quant="bf16", act_scale_fmt="fp32",
                            apply_router_weight_on_input=False, exact=False, tokens=None,
                            return_items=False, w13_bias=None, w2_bias=None,
                            router_weight_in_gemm2=False, act_recipe=None):
    """Form 1: brute-force loop over tokens and slots, no permutation.

    For each (t, i) with e = id[t, i] >= 0: quantise x_t (quantised modes),
    h = W13_e x_t, z = SiLU(h_gate) * h_up, o = W2_e z, y_t += w * o.  The
    same roundings as form 2 are applied item by item (an expert's items are
    stacked as the rows of one matrix product; every step is row-wise).  ``tokens`` restricts
    the tokens evaluated (outputs of different tokens are independent).
    Returns y [len(tokens), H]; with ``return_items`` also the per-item W2
    outputs o [len(tokens), k, H] (zero for skipped slots) and the weights
    w' [len(tokens), k] they were summed with."""
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(topk_ids, dtype=np.int64)
    wts = np.asarray(topk_weights, dtype=np.float64)
    M, k = ids.shape
    tokens = list(range(M)) if tokens is None else list(tokens)
    fmt = _act_scale_fmt(quant, act_scale_fmt)
    w13 = np.asarray(w13)
    w2 = np.asarray(w2)
    H = x.shape[1]
    outs = {}
    # weights are decoded once per expert; the expert's routed items are rows
    # of one matrix, each row put through the steps on its own (quantisation
    # per row, the products row by row in one matrix product)
    experts = sorted({int(ids[t, i]) for t in tokens for i in range(k) if ids[t, i] >= 0})
    for e in experts:
        if quant == "fp8":
            # codes decoded once per expert; the scales enter per K block
            W13 = codecs.e4m3_decode(w13[e])
            W2 = codecs.e4m3_decode(w2[e])
        else:
            W13 = dequant_weights(w13[e][None], None if w13_scale is None else
                                  np.asarray(w13_scale)[e][None], quant)[0]
            W2 = dequant_weights(w2[e][None], None if w2_scale is None else
                                 np.asarray(w2_scale)[e][None], quant)[0]
        I = W2.shape[1]
        its = [(t, i) for t in tokens for i in range(k) if ids[t, i] == e]
        xt = np.stack([x[t] for t, _ in its])
        if apply_router_weight_on_input:
            w_in = np.array([wts[t, i] for t, i in its])
            xt = codecs.round_bf16(codecs.round_fp32(xt * w_in[:, None]))
        if fmt is None:
            h = xt @ W13.T
        else:
            q, s = quant_act_1x128(xt, fmt, act_group(quant))
            if quant == "fp8":
                h = _fp8_rows(q, s, W13, np.asarray(w13_scale)[e])
            else:
                h = (q * np.repeat(s, act_group(quant), axis=1)) @ W13.T
        if w13_bias is not None:
            h = h + np.asarray(w13_bias, dtype=np.float64)[e]
        if not exact:
            h = codecs.round_bf16(h)
        z = gated(h[:, :I], h[:, I:], act_recipe)
        if fmt is None:
            if not exact:
                z = codecs.round_bf16(z)
            o = z @ W2.T
        else:
            q, s = quant_act_1x128(z, fmt, act_group(quant))
            if quant == "fp8":
                o = _fp8_rows(q, s, W2, np.asarray(w2_scale)[e])
            else:
                o = (q * np.repeat(s, act_group(quant), axis=1)) @ W2.T
        if w2_bias is not None:
            o = o + np.asarray(w2_bias, dtype=np.float64)[e]
        if router_weight_in_gemm2:
            o = np.array([wts[t, i] for t, i in its])[:, None] * o
        if not exact:
            o = codecs.round_bf16(o)
        for j, ti in enumerate(its):
            outs[ti] = o[j]
    y = np.zeros((len(tokens), H))
    items = np.zeros((len(tokens), k, H))
    used_w = np.zeros((len(tokens), k))
    for j, t in enumerate(tokens):
        for i in range(k):                      # slot order
            if ids[t, i] < 0:
                continue
            wi = 1.0 if (apply_router_weight_on_input or router_weight_in_gemm2) else wts[t, i]
            y[j] += wi * outs[(t, i)]
            items[j, i] = outs[(t, i)]
            used_w[j, i] = wi
    y = y if exact else codecs.round_bf16(y)
    return (y, items, used_w) if return_items else y


def _fp8_rows(qa, sa, qb, w_scale):
    """h[r, n] = sum_kb sa[r, kb] * sb[n/128, kb] * sum_{k in kb} qa[r, k] * qb[n, k]
    for each row r (qa [R, K] e4m3 values, sa [R, K/128]; qb the decoded e4m3
    weight values [N, K], w_scale [N/128, K/128])."""
    N, K = qb.shape
    sb = np.repeat(np.asarray(w_scale, dtype=np.float64), 128, axis=0)[:N]   # [N, K/128]
    h = np.zeros((qa.shape[0], N))
    for kb in range(K // 128):
        ks = slice(kb * 128, (kb + 1) * 128)
        part = qa[:, ks] @ qb[:, ks].T            # exact: products of e4m3 values
        h += sa[:, kb][:, None] * sb[None, :, kb] * part
    return h


def batched_experts(x_b, counts, w13, w2, w13_scale=None, w2_scale=None, *, quant="bf16",
                    act_scale_fmt="fp32"):
    """The BatchedExperts layout (page "fused_moe.py 分析", activation formats:
    [E, max_tokens, K], one buffer per local expert; page "Blackwell 上的
    DeepGEMM FusedMoE（vLLM）", §2.5: the per-expert counts come with the
    dispatch and the experts run a masked grouped GEMM).

    For each expert e and row r < clamp(counts[e], 0, T): y[e, r] = expert e's
    MLP of x[e, r] with the path's roundings -- form 1 with a single slot of
    weight 1 routed to e, whose bf16 output rounding leaves the bf16 W2 output
    unchanged.  No router weight is applied.  Rows past a count are NaN (they
    have no meaning).  Returns y [E, T, H]."""
    x_b = np.asarray(x_b, dtype=np.float64)
    E, T, H = x_b.shape
    y = np.full((E, T, H), np.nan)
    for e in range(E):
        c = min(max(int(counts[e]), 0), T)
        if c == 0:
            continue
        y[e, :c] = fused_experts_per_token(
            x_b[e, :c], np.full((c, 1), e), np.ones((c, 1)), w13, w2, w13_scale, w2_scale,
            quant=quant, act_scale_fmt=act_scale_fmt)
    return y
