"""Shared helpers of the GPU parity tests (not a test module).

Tolerance reading.  The bound for floating-point outputs is
max|err| <= tol * RMS(y_ref), tol = 1e-2 (bf16 path) or 3e-2 (FP8/FP4 paths).
Both sides store intermediates in bf16 (H1, Z, Y2) and round the output to
bf16.  Two correct implementations whose pre-rounding values differ by a few
fp32 ulps still land on adjacent bf16 values for a small fraction of elements,
and at |y| ~ 4-5 RMS a single bf16 ulp is 2-4% of RMS.  So every element may
first use an allowance for one flip at each bf16 storage point that feeds it
-- one ulp of the output plus w_i * ulp(Y2_i) for each routed item of the token
(``flip_allowance``) -- and the rest of its error must be <= tol * RMS.  On top
of that the RMS of the raw error must stay below tol / 3 * RMS, which a
systematic mistake would break.  Indices and copies are compared bit for bit.
"""
from __future__ import annotations

import contextlib
import numpy as np
import torch

BF16_TOL = 1e-2
QUANT_TOL = 3e-2

# (what, stats) of every check_close call, printed at the end of the run by
# the terminal-summary hook in conftest.py, so the log records the plain
# max|err| / RMS of each comparison next to the asserted quantities.
PARITY_LOG = []


def np32(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def ulp_bf16(v):
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.ldexp(1.0, (e - 7).astype(np.int64)), 2.0 ** -133)


def flip_allowance(y_ref, items, weights):
    """Per-element allowance for one bf16 flip of the output and of each
    routed item's stored GEMM2 row: ulp(y) + sum_i |w_i| * ulp(Y2_i).
    items: [T, k, H] oracle Y2 rows (zeros for skipped slots), weights [T, k]."""
    allow = ulp_bf16(y_ref)
    for i in range(items.shape[1]):
        allow = allow + np.abs(weights[:, i])[:, None] * ulp_bf16(items[:, i])
    return allow


def act_allowance(h1_ref, I):
    """Allowance for z = SiLU(g) * u when g or u (bf16) flipped by one ulp:
    ulp(z) + |dz/dg| ulp(g) + |SiLU(g)| ulp(u)."""
    h = np.asarray(h1_ref, dtype=np.float64)
    g, u = h[:, :I], h[:, I:]
    sig = 1.0 / (1.0 + np.exp(-g))
    z = g * sig * u
    dz_dg = np.abs(u * (sig + g * sig * (1.0 - sig)))
    return ulp_bf16(z) + dz_dg * ulp_bf16(g) + np.abs(g * sig) * ulp_bf16(u)


def check_close(gpu, ref, tol, what="", allow=None):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    if ref.size == 0:
        return {}
    err = np.abs(gpu - ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    allow = ulp_bf16(ref) if allow is None else allow
    excess = float(np.max(err - allow))
    rms_err = float(np.sqrt(np.mean(err ** 2)))
    stats = {"max_err_over_rms": float(err.max() / rms), "rms_err_over_rms": rms_err / rms,
             "max_excess_over_rms": excess / rms, "tol": tol, "n": int(ref.size)}
    PARITY_LOG.append((what, stats))
    assert excess <= tol * rms, f"{what}: {stats}"
    assert rms_err <= tol / 3 * rms, f"{what}: {stats}"
    return stats


def to_dev(d, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def oracle_inputs(d):
    """numpy views of a make_inputs() dict for the oracle."""
    return dict(x=np32(d["x"]), topk_ids=np32(d["topk_ids"]), topk_weights=np32(d["topk_weights"]),
                w13=np32(d["w13"]), w2=np32(d["w2"]), w13_scale=np32(d.get("w13_scale")),
                w2_scale=np32(d.get("w2_scale")))


@contextlib.contextmanager
def bf16_gemm_form(form):
    """Run the block with the bf16 and FP8-block GEMMs forced to one form
    ("single": 128 x 256 tiles on one SM, "pairs": 256 x 256 tiles on SM
    pairs, "auto": by size)."""
    import mixture_experts_ffn_align_gb300 as moe
    moe.moe_debug_set_bf16_gemm_form(form)
    try:
        yield
    finally:
        moe.moe_debug_set_bf16_gemm_form("auto")


def cover_tokens(topk_ids, E, n, seed, experts=None, block=128,
                 which=("first", "last_block", "last")):
    """Tokens for a sampled check of a full-size output: for each expert in
    ``experts`` (default: every expert with routed items) the tokens of its
    first routed row ("first"), of the first row of its last padded block
    ("last_block") and of its last live row ("last", the partial block's
    edge), then random other tokens up to ``n`` in all.  Rows and blocks
    follow the oracle's routing (ascending routed item within an expert)."""
    from oracle import routing
    ids = np.asarray(np32(topk_ids))
    M, k = ids.shape
    route = routing.align_permute(ids, E, block)
    sid, offs, cnt = route["sorted_token_ids"], route["expert_offsets"], route["expert_counts"]
    chosen = set()
    for e in (range(E) if experts is None else experts):
        c = int(cnt[e])
        if c == 0:
            continue
        lo = int(offs[e])
        rows = {"first": lo, "last_block": lo + (c - 1) // block * block, "last": lo + c - 1}
        for w in which:
            chosen.add(int(sid[rows[w]]) // k)
    rng = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(M), np.fromiter(chosen, dtype=np.int64))
    extra = max(0, n - len(chosen))
    if extra:
        chosen.update(int(t) for t in rng.choice(rest, min(extra, rest.size), replace=False))
    return np.array(sorted(chosen), dtype=np.int64)
