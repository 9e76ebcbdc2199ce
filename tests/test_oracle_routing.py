"""Pins for oracle/routing.py: a hand-worked fixture, the closed-form bound
worked by hand, a pure-Python brute force, and the pages' invariants."""
import json
import os

import numpy as np
import pytest

from oracle import routing


def _brute_force(ids, E, A):
    """Nested loops straight from the definition: for each expert in order,
    append its items in ascending r, then pad to a multiple of A."""
    M, k = len(ids), len(ids[0])
    R = M * k
    sorted_ids, blocks, inv = [], [], [[-1] * k for _ in range(M)]
    for e in range(E):
        start = len(sorted_ids)
        for r in range(R):
            if ids[r // k][r % k] == e:
                inv[r // k][r % k] = len(sorted_ids)
                sorted_ids.append(r)
        while (len(sorted_ids) - start) % A:
            sorted_ids.append(R)
        blocks += [e] * ((len(sorted_ids) - start) // A)
    return sorted_ids, blocks, inv


def test_hand_worked_fixture(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "routing_hand_worked.json")))
    out = routing.align_permute(np.array(g["topk_ids"]), g["num_experts"], g["block_size"])
    assert out["expert_counts"].tolist() == g["expert_counts"]
    assert out["expert_offsets"].tolist() == g["expert_offsets"]
    assert out["num_tokens_post_padded"] == g["num_tokens_post_padded"]
    assert out["sorted_token_ids"].tolist() == g["sorted_token_ids"]
    assert out["block_expert_ids"].tolist() == g["block_expert_ids"]
    assert out["inv_perm"].tolist() == g["inv_perm"]
    assert routing.m_sum_bound(4, 2, 3, 4) == g["m_sum_bound"]


def test_bound_hand_worked(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "m_sum_bound_workloads.json")))
    for c in g["cases"]:
        assert routing.m_sum_bound(c["M"], c["topk"], c["E"], c["align"]) == c["bound"], c


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    M, k, E = int(rng.integers(0, 9)), int(rng.integers(1, 4)), int(rng.integers(1, 7))
    A = int(rng.choice([1, 2, 4, 8]))
    ids = rng.integers(-1, E, size=(M, k))
    out = routing.align_permute(ids, E, A)
    s, b, inv = _brute_force(ids.tolist(), E, A)
    total = len(s)
    assert out["num_tokens_post_padded"] == total
    assert out["sorted_token_ids"][:total].tolist() == s
    assert np.all(out["sorted_token_ids"][total:] == M * k)
    assert out["block_expert_ids"][: total // A].tolist() == b
    assert np.all(out["block_expert_ids"][total // A:] == -1)
    assert out["inv_perm"].tolist() == inv


@pytest.mark.parametrize("E,A,M,k", [(8, 128, 16, 2), (256, 128, 512, 8), (8, 16, 64, 2),
                                     (3, 64, 1000, 3), (1024, 32, 100, 4)])
def test_invariants(E, A, M, k):
    rng = np.random.default_rng(E * 7 + A)
    ids = rng.integers(-1, E, size=(M, k))
    out = routing.align_permute(ids, E, A)
    R = M * k
    flat = ids.reshape(-1)
    # every valid routed item lands in exactly one row: sum of counts = #valid
    assert out["expert_counts"].sum() == np.count_nonzero(flat >= 0)
    # segments contiguous, in expert order, aligned to A
    off = out["expert_offsets"]
    assert np.all(off % A == 0) and np.all(np.diff(off) >= out["expert_counts"])
    assert np.all(np.diff(off) - out["expert_counts"] < A)
    sid, inv = out["sorted_token_ids"], out["inv_perm"].reshape(-1)
    # inv_perm inverts the permutation on valid items; invalid ids have -1
    assert np.all(sid[inv[flat >= 0]] == np.nonzero(flat >= 0)[0])
    assert np.all(inv[flat < 0] == -1)
    rows = routing.row_expert_ids(out, A)
    live = sid < R
    assert np.all(rows[live] == flat[sid[live]])
    assert np.all(rows[~live] == -1)
    # the bound holds
    assert out["num_tokens_post_padded"] <= routing.m_sum_bound(M, k, E, A)


def test_bound_is_tight():
    # every expert gets exactly one item: each pads to a full block
    E, A = 8, 128
    ids = np.arange(E).reshape(E, 1)
    out = routing.align_permute(ids, E, A)
    assert out["num_tokens_post_padded"] == routing.m_sum_bound(E, 1, E, A) == E * A


def test_empty_and_out_of_range():
    out = routing.align_permute(np.zeros((0, 2), dtype=np.int64), 8, 128)
    assert out["num_tokens_post_padded"] == 0 and out["sorted_token_ids"].size == 0
    with pytest.raises(ValueError):
        routing.align_permute(np.array([[0, 8]]), 8, 128)


def test_block_d():
    assert routing.block_d(4096) == 1024 and routing.block_d(7168) == 1024
    assert routing.block_d(2880) == 64 and routing.block_d(256) == 256
