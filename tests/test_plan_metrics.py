"""plan_metrics (decode_dsa_kv_gb300/runtime.py), the per-request step
counts read off a plan's outputs, against the oracle's plan of the same ids
on pools in several states: a cold pool, a warm one, and a set flooded past
its ways ([GLM] §4.3: one FIFO pointer per set; with more misses than ways in
one step only the last W of them stay)."""
import numpy as np

import oracle
from decode_dsa_kv_gb300.runtime import plan_metrics


def device_layout(plans, k):
    """The oracle's plans in the device's arrays: [B] counts, [B][k] lists."""
    B = len(plans)
    miss_rows = np.zeros(B, np.int32)
    miss_count = np.zeros(B, np.int32)
    miss_ids = np.full((B, k), -7, np.int32)
    install = np.full((B, k), 9, np.uint8)
    for b, p in enumerate(plans):
        M = p.miss_count
        miss_rows[b] = int(np.count_nonzero(p.src_map < 0))
        miss_count[b] = M
        miss_ids[b, :M] = p.miss_ids
        install[b, :M] = p.install_code
    return miss_rows, miss_count, miss_ids, install


def test_counts_match_the_oracles_plan():
    rng = np.random.default_rng(3)
    S, W, k, ctx = 16, 4, 48, 4096
    plans, want = [], []
    for case in range(5):
        tags = np.full(S * W, -1, np.int32)
        ptr = np.zeros(S, np.int32)
        if case >= 1:  # a warm pool: some slots tagged
            for slot in rng.choice(S * W, size=S * W // 2, replace=False):
                tags[slot] = (slot // W) + S * int(rng.integers(0, ctx // S))
        pool_ids = [t for t in tags if t >= 0]
        ids = set(rng.choice(pool_ids, size=min(10, len(pool_ids)), replace=False).tolist()
                  if pool_ids else [])
        if case >= 3:  # flood set 5 (and at case 4 also set 9) past its ways
            for s in ([5] if case == 3 else [5, 9]):
                ids |= {s + S * int(j) for j in rng.choice(ctx // S, size=2 * W + 1, replace=False)}
        while len(ids) < k:
            ids.add(int(rng.integers(0, ctx)))
        ids = np.array(sorted(ids)[:k], np.int32)
        p = oracle.dsa_plan(ids, ctx, tags, ptr, S, W)
        plans.append(p)
        sets = p.miss_ids % S
        over = sum(1 for s in np.unique(sets) if np.count_nonzero(sets == s) > W)
        want.append((int(np.count_nonzero(p.src_map >= 0)), p.miss_count,
                     int(np.count_nonzero(p.install)), over))
    got = plan_metrics(*device_layout(plans, k), k=k, S=S)
    assert [w[0] for w in want] == got["hits"]
    assert [w[1] for w in want] == got["misses"]
    assert [w[2] for w in want] == got["installs"]
    assert [w[3] for w in want] == got["overflow_sets"]
    assert got["overflow_sets"][3] >= 1 and got["overflow_sets"][4] >= 2


def test_hits_count_repeated_positions_once_each():
    # a caller's ids may repeat a token: every position that misses counts,
    # the miss list holds it once
    S, W, k = 4, 2, 6
    ids = np.array([3, 3, 8, 8, 8, 12], np.int32)
    tags = np.full(S * W, -1, np.int32)
    tags[0] = 8  # token 8 sits in set 0, way 0
    p = oracle.dsa_plan(ids, 64, tags, np.zeros(S, np.int32), S, W)
    got = plan_metrics(*device_layout([p], k), k=k, S=S)
    assert got["hits"] == [3] and got["misses"] == [2]


def test_without_installs():
    got = plan_metrics([5], [3], np.zeros((1, 8), np.int32), None, k=8, S=4)
    assert got == {"hits": [3], "misses": [3], "installs": None, "overflow_sets": None}
