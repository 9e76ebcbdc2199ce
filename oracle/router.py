"""Router: scores -> top-k experts per token -- oracle.

Test infrastructure only.  Follows the page "fused_moe.py 分析", section
"topk_ids, topk_weights 的由来以及内容" (fused_topk): the router logits
[M, E] are turned into per-expert scores by softmax over the E experts or by
an element-wise sigmoid ("scoring_func"), the k highest-scoring experts of
each token are kept, and with "renormalize" their weights are divided by
their sum; outputs are topk_weights [M, k] fp32, topk_ids [M, k] int32 and
token_expert_indices [M, k] int32.  The expert map (same page, the
expert_map argument of fused_experts, and its worked example
[0, -1, 1, 2, -1, 3, 4, 5]) sends a global expert id to its local id on this
expert-parallel shard, or -1 when the expert lives elsewhere.

Readings where the pages are silent:
* selection: both scoring functions are strictly increasing in the logit, so
  the k highest scores are the k highest logits; the oracle selects on the
  logits themselves (exact inputs, no rounding decides the choice), highest
  first, equal logits in ascending expert order;
* the weights are the selected experts' scores; with renormalize each is
  divided by the sum of the k selected scores;
* token_expert_indices[t, i] = t*k + i, the routed-item index used by the
  routing stage (the page gives the tensor but not its contents);
* the expert map is applied to the selected ids after selection; weights are
  kept, so a token's weights still sum to 1 over all shards.
"""
from __future__ import annotations

import numpy as np


def select_topk(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices [M, k] of the k largest logits per row, largest first; equal
    logits in ascending index order."""
    logits = np.asarray(logits)
    M, E = logits.shape
    out = np.empty((M, k), dtype=np.int32)
    for t in range(M):
        # sort key: (-logit, index); lexsort takes the last key as primary
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))
        out[t] = order[:k]
    return out


def scores(logits: np.ndarray, scoring: str) -> np.ndarray:
    """Per-expert scores in fp64: softmax over the row, or sigmoid."""
    x = np.asarray(logits, dtype=np.float64)
    if scoring == "softmax":
        z = np.exp(x - x.max(axis=1, keepdims=True))
        return z / z.sum(axis=1, keepdims=True)
    if scoring == "sigmoid":
        return 1.0 / (1.0 + np.exp(-x))
    raise ValueError(scoring)


def topk_router(logits: np.ndarray, k: int, renormalize: bool = True,
                scoring: str = "softmax", expert_map: np.ndarray | None = None):
    """Returns (topk_weights [M,k] fp64, topk_ids [M,k] int32,
    token_expert_indices [M,k] int32)."""
    logits = np.asarray(logits)
    M, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    ids = select_topk(logits, k)
    s = scores(logits, scoring)
    w = np.take_along_axis(s, ids.astype(np.int64), axis=1)
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    if expert_map is not None:
        emap = np.asarray(expert_map, dtype=np.int32)
        if emap.shape != (E,):
            raise ValueError("expert_map must have one entry per expert")
        ids = emap[ids]
    tei = (np.arange(M, dtype=np.int32)[:, None] * k
           + np.arange(k, dtype=np.int32)[None, :]).astype(np.int32)
    return w, ids.astype(np.int32), tei
