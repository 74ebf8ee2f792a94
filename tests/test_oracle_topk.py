"""Pins of the oracle's top-k (indexer selection, GLM-5.2 shared-Indexer KV
Cache Offload page §2.1) against brute force and invariants."""
import itertools

import numpy as np
import pytest

from oracle import topk_ids


def _beats(s, i, j):
    """Position i ranks above position j: larger score, then lower index."""
    a, b = float(s[i]) + 0.0, float(s[j]) + 0.0
    return a > b or (a == b and i < j)


def _brute(s, k):
    """Every k-subset that dominates its complement; must be exactly one."""
    n = len(s)
    found = []
    for sub in itertools.combinations(range(n), k):
        rest = [j for j in range(n) if j not in sub]
        if all(_beats(s, i, j) for i in sub for j in rest):
            found.append(sub)
    assert len(found) == 1
    return np.array(found[0], dtype=np.int32)


def test_brute_force_tiny_all_k():
    rng = np.random.default_rng(5)
    values = np.array([0.0, -0.0, 0.5, 1.0, -1.0, np.inf, -np.inf, 0.25], np.float32)
    for trial in range(60):
        n = int(rng.integers(1, 9))
        s = values[rng.integers(0, len(values), n)] if trial % 2 else \
            rng.standard_normal(n).astype(np.float32)
        for k in range(1, n + 1):
            assert np.array_equal(topk_ids(s, n, k), _brute(s, k)), (s, k)


def test_invariants_large():
    rng = np.random.default_rng(6)
    s = np.round(rng.standard_normal(5000) * 4) / 4       # many exact ties
    s = s.astype(np.float32)
    k = 300
    ids = topk_ids(s, 5000, k)
    assert ids.size == k and np.all(np.diff(ids) > 0)
    sel = np.zeros(5000, bool)
    sel[ids] = True
    thr = s[ids].min()
    assert np.all(s[~sel] <= thr)
    # ties at the threshold: every selected tie has a lower index than every
    # unselected tie
    tie_sel = np.flatnonzero(sel & (s == thr))
    tie_out = np.flatnonzero(~sel & (s == thr))
    if tie_out.size:
        assert tie_sel.max() < tie_out.min()


def test_signed_zero_is_one_score():
    assert topk_ids(np.array([-0.0, 0.0], np.float32), 2, 1).tolist() == [0]
    assert topk_ids(np.array([0.0, -0.0], np.float32), 2, 1).tolist() == [0]


def test_all_equal_takes_lowest_positions():
    assert topk_ids(np.full(50, 3.0, np.float32), 50, 7).tolist() == list(range(7))


def test_context_bound_and_nan():
    s = np.array([0.0, 1.0, 2.0, 9.0], np.float32)
    assert topk_ids(s, 3, 2).tolist() == [1, 2]          # position 3 is past the context
    with pytest.raises(ValueError):
        topk_ids(np.array([np.nan, 1.0], np.float32), 2, 1)
    with pytest.raises(ValueError):
        topk_ids(s, 2, 3)
