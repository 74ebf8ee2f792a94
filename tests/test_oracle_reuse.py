"""Pins of the adjacent-step reuse plan (oracle/reuse.py) against things other
than itself: a brute-force search, the step identity (a repeated selection is
all hits), disjoint selections (all misses), and the served bytes."""
import numpy as np
import pytest

import oracle
from oracle.reuse import plan_reuse


def brute(ids, prev, n):
    out = []
    for t in ids:
        hit = [j for j, u in enumerate(prev) if u == t]
        out.append(hit[0] if hit else -1 - t)
    return np.array(out, np.int32)


@pytest.mark.parametrize("seed", range(6))
def test_against_brute_force(seed):
    rng = np.random.default_rng(seed)
    n, k = 200, 40
    prev = np.sort(rng.choice(n, k, replace=False))
    ids = np.sort(rng.choice(n, k, replace=False))
    p = plan_reuse(ids, prev, n)
    assert np.array_equal(p.src_map, brute(ids, prev, n))
    miss = [int(t) for t in ids if t not in set(prev.tolist())]
    assert p.miss_ids.tolist() == sorted(miss)
    assert all(ids[j] == t for t, j in zip(p.miss_ids, p.miss_pos))
    assert p.miss_count + int(np.sum(p.src_map >= 0)) == k


def test_same_selection_is_all_hits_and_served_in_place():
    ids = np.array([3, 8, 9, 20, 41], np.int32)
    p = plan_reuse(ids, ids, 50)
    assert p.src_map.tolist() == [0, 1, 2, 3, 4] and p.miss_count == 0


def test_disjoint_or_empty_previous_is_all_misses():
    ids = np.array([1, 5, 7], np.int32)
    for prev in (np.array([2, 4, 6], np.int32), np.full(3, -1, np.int32)):
        p = plan_reuse(ids, prev, 10)
        assert p.src_map.tolist() == [-2, -6, -8]
        assert p.miss_ids.tolist() == [1, 5, 7] and p.miss_pos.tolist() == [0, 1, 2]


def test_served_rows_equal_the_host_rows():
    # serving through the plan (previous buffer for hits, host rows for misses)
    # gives exactly the host rows of the current ids
    rng = np.random.default_rng(9)
    n, k = 300, 25
    host = rng.integers(0, 65536, size=(n, 4), dtype=np.uint16)
    prev = np.sort(rng.choice(n, k, replace=False))
    prev_buf = host[prev]
    ids = np.sort(np.concatenate([prev[:10], rng.choice(np.setdiff1d(np.arange(n), prev), k - 10,
                                                        replace=False)]))
    p = plan_reuse(ids, prev, n)
    got = np.stack([prev_buf[s] if s >= 0 else host[-1 - s] for s in p.src_map])
    assert np.array_equal(got, host[ids])


def test_rejects_ids_outside_the_context():
    with pytest.raises(ValueError):
        plan_reuse(np.array([5, 12]), np.array([1, 2]), 10)


def test_exported():
    assert oracle.plan_reuse is plan_reuse
