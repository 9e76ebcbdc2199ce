"""Block-aligned routing (moe_align_block_size / ep_scatter) -- oracle.

Test infrastructure only.  Follows the page "fused_moe.py 分析", section
"moe_align_block_size 的作用": every (token, top-k slot) pair is a routed item,
items are sorted by expert, and each expert's count is padded up to a multiple
of the block size; the outputs are ``sorted_token_ids``, one expert id per
block and ``num_tokens_post_padded``.  The inverse permutation ``inv_perm``
[M, k] and the per-expert segment starts come from the page "Blackwell 上的
DeepGEMM FusedMoE（vLLM）", §2.6.2 (ep_scatter_1: rounded prefix sum per expert;
ep_scatter_2: each item writes its destination row into inv_perm; ids < 0 are
skipped).  The buffer bound is §2.6.1 (compute_aligned_M_and_alignment).

Readings where the pages are silent:
* routed item r = t*k + i, so its token is r // k (the page "fused_moe.py 分析",
  "构造 A / B 指针": A is addressed by offs_token // top_k);
* within an expert, items keep ascending r (stable; §2.6.2 says segments are
  "in token order");
* padding entries of sorted_token_ids hold R = M*k (any value >= R is padding);
* block ids past the used blocks are -1; experts with no items get no block;
  segments are laid out in ascending expert order;
* ids < 0 are skipped (no row, inv_perm = -1).
"""
from __future__ import annotations

import numpy as np


def round_up(a: int, b: int) -> int:
    return (a + b - 1) // b * b


def m_sum_bound(M: int, topk: int, num_experts: int, block_size: int) -> int:
    """Worst-case padded row count, the closed form of
    compute_aligned_M_and_alignment when per-expert counts are unknown on the
    host (page "Blackwell 上的 DeepGEMM FusedMoE（vLLM）", §2.6.1):
    round_up(M*k + min(M*k, E) * (align - 1), align)."""
    R = M * topk
    return round_up(R + min(R, num_experts) * (block_size - 1), block_size)


def align_permute(topk_ids, num_experts: int, block_size: int):
    """Routing half of the permute.

    topk_ids: [M, k] integer array, -1 = invalid slot; values >= num_experts
    are rejected.  Returns a dict of numpy int64 arrays:
      expert_counts [E], expert_offsets [E+1] (padded segment starts),
      sorted_token_ids [M_sum_bound] (routed item index r, padding = R),
      block_expert_ids [M_sum_bound / block_size] (-1 past the end),
      num_tokens_post_padded (int), inv_perm [M, k] (-1 for invalid slots).
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    M, k = ids.shape
    R = M * k
    E, A = num_experts, block_size
    if np.any(ids >= E):
        raise ValueError("expert id out of range")
    flat = ids.reshape(-1)
    counts = np.bincount(flat[flat >= 0], minlength=E)[:E]
    padded = np.array([round_up(int(c), A) for c in counts], dtype=np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    total = int(offsets[E])
    cap = m_sum_bound(M, k, E, A)
    assert total <= cap
    sorted_ids = np.full(cap, R, dtype=np.int64)
    block_ids = np.full(cap // A, -1, dtype=np.int64)
    inv_perm = np.full(R, -1, dtype=np.int64)
    valid = np.nonzero(flat >= 0)[0]
    # stable sort of the valid items by expert: ascending r inside an expert
    order = valid[np.argsort(flat[valid], kind="stable")]
    fill = offsets[:E].copy()
    for r in order:
        e = flat[r]
        sorted_ids[fill[e]] = r
        inv_perm[r] = fill[e]
        fill[e] += 1
    for e in range(E):
        block_ids[offsets[e] // A: offsets[e + 1] // A] = e
    return {
        "expert_counts": counts.astype(np.int64),
        "expert_offsets": offsets,
        "sorted_token_ids": sorted_ids,
        "block_expert_ids": block_ids,
        "num_tokens_post_padded": total,
        "inv_perm": inv_perm.reshape(M, k),
    }


def row_expert_ids(route, block_size: int):
    """Per-row expert id (DeepGEMM's m_indices, page "Blackwell 上的 DeepGEMM
    FusedMoE（vLLM）", §2.6.2): the block's expert for filled rows, -1 for
    padding rows and rows past num_tokens_post_padded."""
    R = len(route["inv_perm"].reshape(-1))
    rows = np.repeat(route["block_expert_ids"], block_size)
    return np.where(route["sorted_token_ids"] < R, rows, -1)


def block_d(H: int) -> int:
    """Column tile of ep_gather (same page, §2.6.5): gcd(H, 1024)."""
    return int(np.gcd(H, 1024))
