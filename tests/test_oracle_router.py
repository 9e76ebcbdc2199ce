"""Pins for oracle/router.py: hand-worked fixtures (closed-form softmax and
sigmoid values, a tie, the pages' expert-map example), SciPy's softmax and
logistic functions, a pure-Python selection brute force, and invariants."""
import json
import os

import numpy as np
import pytest
from scipy import special

from oracle import router


@pytest.fixture(scope="module")
def gold(golden_dir):
    with open(os.path.join(golden_dir, "router_hand_worked.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("scoring", ["softmax", "sigmoid"])
def test_hand_worked_scores(gold, scoring):
    g = gold[scoring]
    x = np.array(g["logits"])
    w, ids, tei = router.topk_router(x, g["k"], renormalize=True, scoring=scoring)
    assert ids.tolist() == g["topk_ids"]
    np.testing.assert_allclose(w, g["topk_weights_renorm"], rtol=1e-14)
    w_raw, ids_raw, _ = router.topk_router(x, g["k"], renormalize=False, scoring=scoring)
    assert ids_raw.tolist() == g["topk_ids"]
    np.testing.assert_allclose(w_raw, g["topk_weights_raw"], rtol=1e-14)
    assert tei.tolist() == [[0, 1]]


def test_hand_worked_tie_order(gold):
    g = gold["ties"]
    _, ids, _ = router.topk_router(np.array(g["logits"]), g["k"])
    assert ids.tolist() == g["topk_ids"]


def test_pages_expert_map_example(gold):
    g = gold["expert_map"]
    emap = np.array(g["map"], dtype=np.int32)
    # logits that select exactly the fixture's global ids, in that order
    gl = np.array(g["global_ids"])
    x = np.full((len(gl), len(emap)), -5.0)
    for t, row in enumerate(gl):
        for i, e in enumerate(row):
            x[t, e] = 3.0 - i
    w0, ids0, _ = router.topk_router(x, gl.shape[1])
    assert ids0.tolist() == g["global_ids"]
    w, ids, _ = router.topk_router(x, gl.shape[1], expert_map=emap)
    assert ids.tolist() == g["local_ids"]
    np.testing.assert_array_equal(w, w0)          # weights are not touched by the map


def _brute_select(row, k):
    """Selection by repeated scans: take the largest remaining logit, the
    lowest index among equals, k times."""
    taken, out = set(), []
    for _ in range(k):
        best = None
        for e, v in enumerate(row):
            if e in taken:
                continue
            if best is None or v > row[best]:
                best = e
        taken.add(best)
        out.append(best)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_selection_against_brute_force(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(2, 9))
    k = int(rng.integers(1, E + 1))
    # few distinct values so that ties are frequent
    x = rng.integers(-2, 3, size=(20, E)).astype(np.float64)
    ids = router.select_topk(x, k)
    for t in range(x.shape[0]):
        assert ids[t].tolist() == _brute_select(list(x[t]), k)


@pytest.mark.parametrize("scoring", ["softmax", "sigmoid"])
def test_weights_match_scipy(scoring):
    rng = np.random.default_rng(3)
    x = rng.normal(size=(50, 32)) * 2
    w, ids, _ = router.topk_router(x, 6, renormalize=False, scoring=scoring)
    full = special.softmax(x, axis=1) if scoring == "softmax" else special.expit(x)
    np.testing.assert_allclose(w, np.take_along_axis(full, ids.astype(np.int64), 1), rtol=1e-13)
    wr, _, _ = router.topk_router(x, 6, renormalize=True, scoring=scoring)
    sel = np.take_along_axis(full, ids.astype(np.int64), 1)
    np.testing.assert_allclose(wr, sel / sel.sum(1, keepdims=True), rtol=1e-13)


def test_invariants():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(200, 64)).astype(np.float32)
    for scoring in ("softmax", "sigmoid"):
        w, ids, tei = router.topk_router(x, 8, scoring=scoring)
        np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-12)
        assert np.all(np.diff(w, axis=1) <= 0)                 # largest score first
        assert all(len(set(r)) == 8 for r in ids.tolist())     # distinct experts
        assert ids.min() >= 0 and ids.max() < 64
        assert tei.tolist() == [[t * 8 + i for i in range(8)] for t in range(200)]
    # k = E keeps every expert; softmax weights are then the softmax itself
    w, ids, _ = router.topk_router(x[:5], 64, renormalize=False)
    np.testing.assert_allclose(np.sort(w, 1), np.sort(special.softmax(x[:5].astype(np.float64), 1), 1),
                               rtol=1e-12)


def test_bad_arguments():
    with pytest.raises(ValueError):
        router.topk_router(np.zeros((2, 4)), 5)
    with pytest.raises(ValueError):
        router.topk_router(np.zeros((2, 4)), 2, scoring="relu")
    with pytest.raises(ValueError):
        router.topk_router(np.zeros((2, 4)), 2, expert_map=np.zeros(3, np.int32))
