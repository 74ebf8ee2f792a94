"""Pins of the oracle's DsaPlan / metadata update (GLM-5.2 shared-Indexer KV
Cache Offload page, §4.2 shared planning, §4.3 set-associative FIFO, §5)."""
import numpy as np
import pytest

from oracle import dsa_plan, metadata_update


def fifo_simulate(ids, tags, ptr, S, W):
    """A literal set-associative cache with one round-robin pointer per set,
    driven one token at a time: look every id up against the cache as it was
    at the start of the step, then install the distinct misses one by one in
    ascending id, each into the slot under its set's pointer, advancing that
    pointer by one per install. Returns (hits, slot of every install in order,
    final tags, final pointers)."""
    tags = list(tags)
    ptr = list(ptr)
    start = list(tags)
    hits = {}
    misses = set()
    for t in ids:
        s = t % S
        ways = [w for w in range(W) if start[s * W + w] == t]
        if ways:
            hits[t] = s * W + ways[0]
        else:
            misses.add(t)
    slots = []
    for t in sorted(misses):
        s = t % S
        slot = s * W + ptr[s]
        tags[slot] = t
        ptr[s] = (ptr[s] + 1) % W
        slots.append(slot)
    return hits, slots, tags, ptr


def _check_against_simulator(ids, ctx, tags, ptr, S, W):
    plan = dsa_plan(ids, ctx, tags, ptr, S, W)
    hits, slots, tags_end, ptr_end = fifo_simulate(ids, tags, ptr, S, W)
    # per-position source
    for j, t in enumerate(ids):
        if t in hits:
            assert plan.src_map[j] == hits[t]
        else:
            assert plan.src_map[j] == -1 - t
    # miss list, first positions, victims
    assert plan.miss_ids.tolist() == sorted({t for t in ids if t not in hits})
    for t, p in zip(plan.miss_ids, plan.miss_pos):
        assert ids[p] == t and t not in ids[:p]
    assert plan.victim.tolist() == slots
    # install flags: the miss is still in its slot at the end of the sequence
    for t, v, keep in zip(plan.miss_ids, plan.victim, plan.install):
        assert bool(keep) == (tags_end[v] == t)
    # metadata update reproduces the simulated cache
    t2 = np.array(tags, np.int32)
    p2 = np.array(ptr, np.int32)
    metadata_update(t2, p2, plan)
    assert t2.tolist() == tags_end and p2.tolist() == ptr_end
    return plan


def test_hand_worked_overflow():
    # S = 2 sets of W = 2 ways. Set 0 holds tokens 4 (way 0) and 6 (way 1),
    # pointer at way 1; set 1 holds token 1 in way 0, way 1 empty, pointer at
    # way 1 (the state a cold pool reaches after installing token 1).
    S, W = 2, 2
    tags = [4, 6, 1, -1]
    ptr = [1, 1]
    ids = [0, 1, 2, 4, 8, 10, 12, 3]
    plan = _check_against_simulator(ids, 16, tags, ptr, S, W)
    # hits: 1 -> slot 2, 4 -> slot 0; misses encoded -1 - t
    assert plan.src_map.tolist() == [-1, 2, -3, 0, -9, -11, -13, -4]
    # misses ascending: 0 2 3 8 10 12, first positions 0 2 7 4 5 6
    assert plan.miss_ids.tolist() == [0, 2, 3, 8, 10, 12]
    assert plan.miss_pos.tolist() == [0, 2, 7, 4, 5, 6]
    # set 0 takes five misses (ranks 0..4) from pointer 1: ways 1 0 1 0 1;
    # set 1 takes one miss from pointer 1: way 1 -> slot 3
    assert plan.victim.tolist() == [1, 0, 3, 1, 0, 1]
    # only the last W = 2 misses of set 0 survive (10 and 12); 3 is installed
    assert plan.install.tolist() == [False, False, True, False, True, True]
    assert plan.ptr_next.tolist() == [0, 0]
    t2, p2 = np.array(tags, np.int32), np.array(ptr, np.int32)
    metadata_update(t2, p2, plan)
    # token 4 was a hit this step and is still evicted (plain FIFO)
    assert t2.tolist() == [10, 12, 1, 3] and p2.tolist() == [0, 0]


def test_duplicates_listed_once():
    S, W = 4, 2
    tags = [-1] * 8
    tags[1 * 2 + 0] = 5
    ids = [9, 5, 9, 13, 5, 9]
    plan = _check_against_simulator(ids, 20, tags, [1, 1, 0, 0], S, W)
    assert plan.src_map.tolist() == [-10, 2, -10, -14, 2, -10]
    assert plan.miss_rows == 4                      # 9 three times, 13 once
    assert plan.miss_ids.tolist() == [9, 13]
    assert plan.miss_pos.tolist() == [0, 3]


def test_random_sequences_against_simulator():
    rng = np.random.default_rng(11)
    for trial in range(40):
        S = int(rng.choice([1, 2, 3, 8]))
        W = int(rng.choice([1, 2, 4]))
        ctx = int(rng.integers(8, 64))
        tags = [-1] * (S * W)
        ptr = [0] * S
        for step in range(5):
            k = int(rng.integers(1, ctx + 1))
            ids = sorted(rng.choice(ctx, size=k, replace=False).tolist())
            if trial % 3 == 0:                       # unsorted, with repeats
                ids = rng.choice(ids, size=k + 3).tolist()
            plan = _check_against_simulator(ids, ctx, tags, ptr, S, W)
            assert plan.miss_count + sum(1 for s in plan.src_map if s >= 0) >= len(set(ids))
            t2, p2 = np.array(tags, np.int32), np.array(ptr, np.int32)
            metadata_update(t2, p2, plan)
            tags, ptr = t2.tolist(), p2.tolist()
            # invariants: pointers in range, tags unique within a set and in
            # their own set
            assert all(0 <= p < W for p in ptr)
            for s in range(S):
                held = [t for t in tags[s * W:(s + 1) * W] if t >= 0]
                assert len(held) == len(set(held))
                assert all(t % S == s for t in held)


def test_hits_plus_misses_is_k_for_distinct_ids():
    rng = np.random.default_rng(3)
    S, W, ctx, k = 16, 4, 400, 96
    tags = [-1] * (S * W)
    ptr = [0] * S
    for _ in range(6):
        ids = np.sort(rng.choice(ctx, k, replace=False))
        plan = dsa_plan(ids, ctx, tags, ptr, S, W)
        hits = int((plan.src_map >= 0).sum())
        assert hits + plan.miss_count == k
        assert np.all(np.diff(plan.miss_ids) > 0)
        t2, p2 = np.array(tags, np.int32), np.array(ptr, np.int32)
        metadata_update(t2, p2, plan)
        tags, ptr = t2.tolist(), p2.tolist()


def test_rejects_bad_input():
    with pytest.raises(ValueError):
        dsa_plan([3, 40], 20, [-1] * 4, [0, 0], 2, 2)      # id past the context
    with pytest.raises(ValueError):
        dsa_plan([3], 20, [-1] * 4, [0, 2], 2, 2)          # pointer >= W


def test_install_code_orders_installs_around_hit_reads():
    """install_code splits the installs into those that may land before the
    step's hits are read (1) and those that must wait for the reads (2):
    writing the 1s first, then reading every hit, then writing the 2s serves
    every hit its own token and leaves the simulator's final cache. Writing
    all installs before the reads breaks a hit in some of these steps, so the
    split is needed (the page: each layer reads its rows before its own refill,
    §4.4)."""
    rng = np.random.default_rng(23)
    needed = 0
    for trial in range(60):
        S = int(rng.choice([1, 2, 4]))
        W = int(rng.choice([1, 2, 4]))
        ctx = int(rng.integers(8, 48))
        tags = [-1] * (S * W)
        ptr = [0] * S
        for step in range(6):
            k = int(rng.integers(1, ctx + 1))
            ids = sorted(rng.choice(ctx, size=k, replace=False).tolist())
            plan = dsa_plan(ids, ctx, tags, ptr, S, W)
            code = plan.install_code
            assert code.tolist() == [0 if not keep else code[i] for i, keep in enumerate(plan.install)]
            _, _, tags_end, ptr_end = fifo_simulate(ids, tags, ptr, S, W)
            for order in ("split", "all_first"):
                pool = list(tags)               # a slot's row is its token
                for t, v, c in zip(plan.miss_ids, plan.victim, code):
                    if c == 1 or (order == "all_first" and c == 2):
                        pool[v] = int(t)
                served = [pool[s] == t for s, t in zip(plan.src_map, ids) if s >= 0]
                if order == "split":
                    assert all(served), (trial, step)
                    for t, v, c in zip(plan.miss_ids, plan.victim, code):
                        if c == 2:
                            pool[v] = int(t)
                    assert pool == tags_end
                elif not all(served):
                    needed += 1
                    assert any(c == 2 for c in code)
            tags, ptr = tags_end, ptr_end
    assert needed > 0
