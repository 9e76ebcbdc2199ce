"""moe_align_permute_noalloc: the routing + permute stage for callers that may
not allocate device memory when they call the library (for example a serving
engine that reserves the device for its own memory pool).  Its scratch is a
fixed array inside the library instead of a caller workspace.

The check: two calls in a row through the C ABI, on two different problems,
each compared with the workspace-taking moe_align_permute on the same inputs.
Indices and permuted rows are compared bit for bit (the tolerance the other
stage-1 tests use).  Both problems are large enough to route in several CTAs,
the path that keeps its per-segment histograms in the shared array (a small
problem routes in one CTA with its histograms in shared memory).  The second
has fewer segments and experts than the first, so stale histogram contents
left in the array by the first call would show.  This file is named to be
collected last."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_align_gb300 as moe
from moe_synth import CONFIGS, MoEConfig, make_inputs

pytestmark = pytest.mark.gpu

OUTPUTS = ("sorted_ids", "block_expert_ids", "expert_offsets", "num_post_padded", "inv_perm")


def _stage1(p, d, noalloc):
    b = moe.stage_buffers(p)
    for k in OUTPUTS + ("x_perm",):
        b[k].fill_(-7 if b[k].dtype == torch.int32 else 0)
    args = (p, d["x"], d["topk_ids"], None, b["sorted_ids"], b["block_expert_ids"],
            b["expert_offsets"], b["num_post_padded"], b["inv_perm"], b["x_perm"],
            b["x_perm_scale"])
    if noalloc:
        moe.moe_align_permute_noalloc(*args)
    else:
        moe.moe_align_permute(*args, b["align_ws"])
    assert moe.moe_sync_status() == 0
    return b


def _compare(p, d):
    got = _stage1(p, d, noalloc=True)
    ref = _stage1(p, d, noalloc=False)
    for k in OUTPUTS:
        assert torch.equal(got[k], ref[k]), k
    n = int(ref["num_post_padded"].item())
    assert torch.equal(got["x_perm"][:n], ref["x_perm"][:n])
    if ref["x_perm_scale"] is not None:
        assert torch.equal(got["x_perm_scale"][:n], ref["x_perm_scale"][:n])


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    big = CONFIGS["dsfp8"]                       # 128 segments x 256 experts, FP8 permute
    # 32 segments x 128 experts: 16384 routed items take the multi-CTA routing
    # too, and read a smaller corner of the array the first call filled
    small = MoEConfig("small", M=2048, H=512, I=256, E=128, topk=8, quant="bf16",
                      routing="softmax", seed=71, invalid_frac=0.1)
    # three routing kernels (histograms, scan, scatter) + the permute
    assert moe.moe_align_permute_launches(moe.Problem.from_config(small)) == 4
    assert moe.moe_align_workspace_bytes(moe.Problem.from_config(small)) < \
        moe.moe_align_workspace_bytes(moe.Problem.from_config(big))
    for cfg in (big, small):
        d = make_inputs(cfg, "cuda", weights=False)
        _compare(moe.Problem.from_config(cfg), d)


def test_noalloc_rejects_problems_beyond_its_scratch():
    p = moe.Problem(M=16384, H=128, I=128, E=1024, topk=16)
    assert moe.moe_align_workspace_bytes(p) > moe.NOALLOC_SCRATCH_BYTES
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_align_permute_noalloc(p, None, None, None, None, None, None, None, None, None,
                                      None)
    assert ei.value.status == 5   # MOE_ERR_WORKSPACE_TOO_SMALL, nothing enqueued
