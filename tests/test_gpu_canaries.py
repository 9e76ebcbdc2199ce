"""Stray-write checks of every stage (a substitute for a memory checker).

Each output buffer of the staged pipeline is allocated with a tail of extra
rows and bytes past its end and is filled with a sentinel before the calls.
After routing + permute, GEMM1 (plain and with the fused activation), the
activation stage, GEMM2 and the reduce:
  * the tail past every buffer is untouched;
  * the rows of the padded layout at or past num_tokens_post_padded are
    untouched (no stage writes there: the GEMMs and the activation stop at
    the used blocks, the permute zeroes only padding rows below the count);
  * the rows below the count hold values, not the sentinel.
A GEMM block taller than the padding granularity, or a tile count read
wrong, would write into another region (page "Blackwell 上的 DeepGEMM
FusedMoE（vLLM）", §2.6.3: BLOCK_M above the alignment reads another
expert's id).  Every quantisation mode and both GEMM forms run on ragged
expert loads (empty experts, one row, a block edge, a partial last block)."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import MoEConfig, make_inputs

from .gpu_util import bf16_gemm_form

pytestmark = pytest.mark.gpu

TAIL_ROWS = 128
TAIL_BYTES = 256
SENTINEL = 0x5A          # byte pattern of every canary


def _guarded(shape, dtype, device="cuda"):
    """A tensor of `shape` whose storage runs on for TAIL_ROWS rows and
    TAIL_BYTES bytes, everything filled with the sentinel byte; returns
    (view, raw bytes, byte size of the view)."""
    rows = shape[0]
    row_elems = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    esize = torch.empty((), dtype=dtype).element_size()
    nbytes = rows * row_elems * esize
    raw = torch.full((nbytes + TAIL_ROWS * row_elems * esize + TAIL_BYTES,), SENTINEL,
                     dtype=torch.uint8, device=device)
    view = raw[:nbytes].view(dtype).view(shape)
    return view, raw, nbytes


def _buffers(p):
    ref = moe.stage_buffers(p)
    out = {}
    for k, t in ref.items():
        if t is None or k == "align_ws":
            out[k] = (t, None, 0)
        else:
            out[k] = _guarded(tuple(t.shape), t.dtype)
    return out


def _ragged(quant, counts, H, I, seed):
    ids = np.concatenate([np.full(c, e, dtype=np.int32) for e, c in enumerate(counts)])
    np.random.default_rng(seed).shuffle(ids)
    M = len(ids)
    fmt = "ue8m0" if quant in ("mxfp4", "mxfp8") else "fp32"
    cfg = MoEConfig("canary", M=M, H=H, I=I, E=len(counts), topk=1, quant=quant,
                    routing="softmax", seed=seed, act_scale_fmt=fmt)
    d = make_inputs(cfg, "cuda")
    d["topk_ids"] = torch.from_numpy(ids).view(M, 1).cuda()
    return cfg, d


def _check(bufs, n, padded_keys):
    for k, (view, raw, nbytes) in bufs.items():
        if raw is None:
            continue
        tail = raw[nbytes:]
        assert bool((tail == SENTINEL).all()), f"{k}: write past the end of the buffer"
        if k in padded_keys:
            rows = view.shape[0]
            row_bytes = nbytes // rows
            past = raw[n * row_bytes:nbytes]
            assert bool((past == SENTINEL).all()), f"{k}: write at or past row {n}"


CASES = [("bf16", "single"), ("bf16", "pairs"), ("fp8", "single"), ("fp8", "pairs"),
         ("mxfp4", "auto"), ("mxfp8", "auto")]


@pytest.mark.parametrize("quant,form", CASES)
@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("bs", [128, 32])
def test_no_stage_writes_outside_its_rows(quant, form, fuse, bs):
    # bf16 GEMM2 tiles are 256 columns wide (H % 256 == 0); the quantised
    # GEMMs take H = 640, a 128-wide last column tile
    counts, H, I = [0, 1, 127, 128, 129, 300, 0], (512 if quant == "bf16" else 640), 256
    cfg, d = _ragged(quant, counts, H, I, 31)
    p = moe.Problem.from_config(cfg, block_size=bs)
    bufs = _buffers(p)
    b = {k: v[0] for k, v in bufs.items()}
    b["align_ws"] = torch.empty(max(moe.moe_align_workspace_bytes(p), 1), dtype=torch.uint8,
                                device="cuda")
    q = quant != "bf16"
    with bf16_gemm_form(form):
        moe.moe_align_permute(p, d["x"], d["topk_ids"], None, b["sorted_ids"],
                              b["block_expert_ids"], b["expert_offsets"], b["num_post_padded"],
                              b["inv_perm"], b["x_perm"], b["x_perm_scale"], b["align_ws"])
        if fuse:
            moe.grouped_gemm_w13(p, b["x_perm"], b["x_perm_scale"], d["w13"], d["w13_scale"],
                                 b["block_expert_ids"], b["num_post_padded"], b["z"],
                                 b["z_scale"], fuse_act=True)
        else:
            moe.grouped_gemm_w13(p, b["x_perm"], b["x_perm_scale"], d["w13"], d["w13_scale"],
                                 b["block_expert_ids"], b["num_post_padded"], b["h1"],
                                 None, fuse_act=False)
            moe.act_mul_quant(p, b["h1"], b["num_post_padded"], b["z"], b["z_scale"])
        moe.grouped_gemm_w2(p, b["z"], b["z_scale"], d["w2"], d["w2_scale"],
                            b["block_expert_ids"], b["num_post_padded"], b["y2"])
        moe.unpermute_reduce(p, b["y2"], b["inv_perm"], d["topk_weights"], b["y"])
    assert moe.moe_sync_status() == 0
    n = int(b["num_post_padded"].item())
    assert 0 < n < b["x_perm"].shape[0]
    padded = {"x_perm", "y2", "z"} | ({"x_perm_scale", "z_scale"} if q else set()) | \
             (set() if fuse else {"h1"})
    _check(bufs, n, padded)
    # the used rows were written (the sentinel byte pattern is not a value
    # any of them holds in all of a row's bytes)
    for k in padded:
        view = b[k][:n].contiguous().view(torch.uint8).view(n, -1)
        assert not bool((view == SENTINEL).all(dim=1).any()), f"{k}: a used row was not written"
    # sorted ids and block ids: the routing writes the whole bound (padding
    # and -1 past the used blocks), so only the tails are checked above
