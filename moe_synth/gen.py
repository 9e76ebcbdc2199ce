"""Seeded generators (torch Philox/MT streams, CPU or CUDA) for every input.

Recipe (one seed per workload, see ``configs.CONFIGS``):

* x: N(0, 1) rounded to bf16.
* Router: logits -> softmax -> top-k -> renormalise to sum 1 (fp32 weights,
  int32 ids).  ``softmax``: logits ~ N(0,1).  ``uniform``: the same (uniform in
  expectation).  ``skew``: logits ~ Gumbel(0,1) + b on the first 10% of the
  experts, with b found by bisection so the hot experts take 50% +- 1% of the
  routed items.
* bf16 weights: N(0, 0.02) rounded to bf16, w13 [E, 2I, H] (rows [0, I) gate,
  rows [I, 2I) up), w2 [E, H, I].
* fp8 weights: N(0, 0.02) cast to e4m3fn with one fp32 scale per 128x128 block
  (scale = block amax / 448); codes stored as uint8; scales [E, N/128, K/128].
* mxfp4 weights: E2M1 codes uniform over all 16 codes, packed two per byte
  (low nibble = even k) as [E, N, K/2] uint8; E8M0 scale codes 127 + j with j
  uniform in {-4..0}, one per 32 along K, stored [E, N, K/32] uint8.
"""
from __future__ import annotations

import torch

from .configs import MoEConfig

_HOT_FRAC = 0.10
_HOT_SHARE = 0.50


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _topk_from_logits(logits: torch.Tensor, k: int):
    p = torch.softmax(logits.float(), dim=-1)
    w, ids = torch.topk(p, k, dim=-1)
    w = w / w.sum(dim=-1, keepdim=True)
    return w.float().contiguous(), ids.to(torch.int32).contiguous()


def make_routing(cfg: MoEConfig, device="cpu", seed_offset: int = 0):
    """Returns (topk_weights [M,k] fp32, topk_ids [M,k] int32, info dict)."""
    g = _gen(cfg.seed * 1000 + 17 + seed_offset, device)
    M, E, k = cfg.M, cfg.E, cfg.topk
    info = {}
    if cfg.routing in ("softmax", "uniform"):
        logits = torch.randn(M, E, generator=g, device=device)
        w, ids = _topk_from_logits(logits, k)
    elif cfg.routing == "skew":
        u = torch.rand(M, E, generator=g, device=device).clamp_(1e-12, 1 - 1e-7)
        gumbel = -torch.log(-torch.log(u))
        n_hot = max(1, int(round(_HOT_FRAC * E)))
        hot = torch.zeros(E, device=device)
        hot[:n_hot] = 1.0

        def share(b):
            _, ids_ = _topk_from_logits(gumbel + b * hot, k)
            return (ids_ < n_hot).float().mean().item()

        lo, hi = 0.0, 20.0
        for _ in range(40):
            mid = 0.5 * (lo + hi)
            if share(mid) < _HOT_SHARE:
                lo = mid
            else:
                hi = mid
        b = 0.5 * (lo + hi)
        w, ids = _topk_from_logits(gumbel + b * hot, k)
        info = {"skew_bias": b, "hot_experts": n_hot,
                "hot_share": (ids < n_hot).float().mean().item()}
    else:
        raise ValueError(cfg.routing)
    if cfg.invalid_frac > 0:
        drop = torch.rand(M, k, generator=g, device=device) < cfg.invalid_frac
        ids = torch.where(drop, torch.full_like(ids, -1), ids)
    return w, ids, info


def _bf16_normal(shape, std, g, device):
    return (torch.randn(*shape, generator=g, device=device) * std).to(torch.bfloat16)


def _fp8_block_weights(E, N, K, g, device):
    """N(0,0.02) weights cast to e4m3fn with fp32 scales per 128x128 block."""
    codes = torch.empty(E, N, K, dtype=torch.uint8, device=device)
    scales = torch.empty(E, (N + 127) // 128, (K + 127) // 128, dtype=torch.float32,
                         device=device)
    for e in range(E):
        w = torch.randn(N, K, generator=g, device=device) * 0.02
        wb = w.view(N // 128, 128, K // 128, 128)
        amax = wb.abs().amax(dim=(1, 3)).clamp_min(1e-12)
        s = amax / 448.0
        q = (wb / s[:, None, :, None]).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
        codes[e] = q.view(torch.uint8).view(N, K)
        scales[e] = s
    return codes, scales


def _mxfp4_weights(E, N, K, g, device):
    lo = torch.randint(0, 16, (E, N, K // 2), generator=g, device=device, dtype=torch.int32)
    hi = torch.randint(0, 16, (E, N, K // 2), generator=g, device=device, dtype=torch.int32)
    packed = (lo | (hi << 4)).to(torch.uint8)
    j = torch.randint(-4, 1, (E, N, K // 32), generator=g, device=device, dtype=torch.int32)
    scales = (127 + j).to(torch.uint8)
    return packed, scales


def _mxfp8_weights(E, N, K, g, device):
    """N(0,0.02) weights cast to e4m3fn with one E8M0 scale per 1x32 group
    along K: 2^ceil(log2(amax / 448)), stored as the biased exponent byte."""
    codes = torch.empty(E, N, K, dtype=torch.uint8, device=device)
    scales = torch.empty(E, N, K // 32, dtype=torch.uint8, device=device)
    for e in range(E):
        w = (torch.randn(N, K, generator=g, device=device) * 0.02).view(N, K // 32, 32)
        amax = w.abs().amax(dim=-1).clamp_min(1e-30)
        ex = torch.ceil(torch.log2(amax / 448.0)).clamp_(-127, 127)
        s = torch.exp2(ex)
        q = (w / s[..., None]).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
        codes[e] = q.view(torch.uint8).view(N, K)
        scales[e] = (ex + 127).to(torch.uint8)
    return codes, scales


def make_inputs(cfg: MoEConfig, device="cpu", weights: bool = True):
    """All inputs of one workload as torch tensors on ``device``.

    Returns a dict with x [M,H] bf16, topk_weights [M,k] f32, topk_ids [M,k]
    i32, and (if ``weights``) w13/w2 plus w13_scale/w2_scale for quantised
    modes (None for bf16).
    """
    g = _gen(cfg.seed, device)
    out = {}
    out["x"] = torch.randn(cfg.M, cfg.H, generator=g, device=device).to(torch.bfloat16)
    w, ids, info = make_routing(cfg, device)
    out["topk_weights"], out["topk_ids"], out["routing_info"] = w, ids, info
    if not weights:
        return out
    gw = _gen(cfg.seed * 7919 + 3, device)
    E, H, I = cfg.E, cfg.H, cfg.I
    if cfg.quant == "bf16":
        out["w13"] = _bf16_normal((E, 2 * I, H), 0.02, gw, device)
        out["w2"] = _bf16_normal((E, H, I), 0.02, gw, device)
        out["w13_scale"] = out["w2_scale"] = None
    elif cfg.quant == "fp8":
        out["w13"], out["w13_scale"] = _fp8_block_weights(E, 2 * I, H, gw, device)
        out["w2"], out["w2_scale"] = _fp8_block_weights(E, H, I, gw, device)
    elif cfg.quant == "mxfp4":
        out["w13"], out["w13_scale"] = _mxfp4_weights(E, 2 * I, H, gw, device)
        out["w2"], out["w2_scale"] = _mxfp4_weights(E, H, I, gw, device)
    elif cfg.quant == "mxfp8":
        out["w13"], out["w13_scale"] = _mxfp8_weights(E, 2 * I, H, gw, device)
        out["w2"], out["w2_scale"] = _mxfp8_weights(E, H, I, gw, device)
    else:
        raise ValueError(cfg.quant)
    return out
