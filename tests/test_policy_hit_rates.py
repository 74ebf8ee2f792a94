"""Pool policies compared by hit rate on the same synthetic score process
(GLM-5.2 shared-Indexer KV Cache Offload, §2.2 previous-step reuse, §3 the
8192-entry LRU pool, §4.3 the set-associative FIFO pool, §7.3 its 8K / 16K
sizes). The LRU pool is pinned here against a brute-force reference; the
comparison itself checks the ordering the pages report, on the oracle."""
import numpy as np
import pytest

import oracle
import workload as wl


def lru_brute(steps, entries):
    """Reference LRU: explicit last-use times, smallest time evicted."""
    last, clock, hits = {}, 0, []
    for ids in steps:
        ids = [int(t) for t in ids]
        h = [t for t in ids if t in last]
        hits.append(len(h))
        for t in h:
            clock += 1
            last[t] = clock
        for t in sorted(set(t for t in ids if t not in h)):
            if len(last) >= entries:
                del last[min(last, key=last.get)]
            clock += 1
            last[t] = clock
    return hits


def test_lru_pool_against_brute_force():
    rng = np.random.default_rng(3)
    steps = [rng.choice(60, 12, replace=False) for _ in range(40)]
    pool = oracle.LruPool(20)
    assert [pool.step(s) for s in steps] == lru_brute(steps, 20)


def test_lru_special_cases():
    pool = oracle.LruPool(4)
    assert pool.step([1, 2, 3]) == 0
    assert pool.step([1, 2, 3]) == 3          # everything resident
    assert pool.step([7, 8]) == 0             # evicts the least recent: 1
    assert pool.step([1]) == 0
    assert pool.step([8]) == 1


def hit_rates(w, steps, requests, start):
    """Mean hit rate from step `start` on, per policy, over `requests`."""
    lens = wl.ctx_lens(w)
    stream = wl.ScoreStream(w)
    rates = {"reuse": [], "fifo_8k": [], "fifo_16k": [], "lru_8k": []}
    prev = {b: np.full(w.k, -1) for b in requests}
    fifo = {(b, S): (np.full(S * 16, -1, np.int32), np.zeros(S, np.int32))
            for b in requests for S in (512, 1024)}
    lru = {b: oracle.LruPool(8192) for b in requests}
    for step in range(steps):
        scores = stream.next()
        for b in requests:
            ids = oracle.topk_ids(scores[b], int(lens[b]), w.k)
            r = {"reuse": int(np.sum(oracle.plan_reuse(ids, prev[b], int(lens[b])).src_map >= 0)),
                 "lru_8k": lru[b].step(ids)}
            prev[b] = ids
            for S, name in ((512, "fifo_8k"), (1024, "fifo_16k")):
                tags, ptr = fifo[(b, S)]
                plan = oracle.dsa_plan(ids, int(lens[b]), tags, ptr, S, 16)
                r[name] = int(np.sum(plan.src_map >= 0))
                oracle.metadata_update(tags, ptr, plan)
            if step >= start:
                for name, h in r.items():
                    rates[name].append(h / w.k)
    return {name: float(np.mean(v)) for name, v in rates.items()}


def test_policy_ordering_on_the_decode_batch_score_process():
    # one request of decode_batch, steps 32..63 (the pools full): the pages'
    # ordering holds -- previous-step reuse < FIFO 8K < LRU 8K, and the 16K
    # FIFO pool above the 8K one (measured: 0.601, 0.736, 0.758, 0.791)
    r = hit_rates(wl.DECODE_BATCH, 64, requests=[0], start=32)
    print("hit rates:", {k: round(v, 3) for k, v in r.items()})
    assert r["reuse"] < r["fifo_8k"] < r["lru_8k"]
    assert r["fifo_8k"] < r["fifo_16k"]
    assert 0.55 < r["reuse"] < 0.65


def lru_slots_brute(steps, P, ctx):
    """Slot-level LRU, one use at a time: every hit touched, every miss into
    the slot with the smallest last-use time (empty slots first, lowest
    index). Returns per step (src_map, victims, installs, tags, last_use)."""
    tags, last, clock, out = [-1] * P, [0] * P, 0, []
    for ids in steps:
        ids = [int(t) for t in ids]
        where = {t: s for s, t in enumerate(tags) if t >= 0}
        src = [where[t] if t in where else -1 - t for t in ids]
        for s in src:
            if s >= 0:
                clock += 1
                last[s] = clock
        misses = sorted({t for t in ids if t not in where})
        vict, latest = [], {}
        for i, t in enumerate(misses):
            empty = [s for s in range(P) if tags[s] < 0]
            v = empty[0] if empty else min(range(P), key=lambda s: last[s])
            vict.append(v)
            latest[v] = i
            tags[v] = t
            clock += 1
            last[v] = clock
        inst = [latest[v] == i for i, v in enumerate(vict)]
        out.append((src, vict, inst, list(tags), list(last)))
    return out


@pytest.mark.parametrize("P,k,n", [(20, 12, 60), (16, 12, 40), (8, 12, 30), (64, 16, 200)])
def test_lru_slots_against_brute_force(P, k, n):
    # includes steps missing more tokens than there are free slots (P = 8 and
    # 16 with 12 selected), so same-step installs evict each other
    rng = np.random.default_rng(P * 100 + k)
    steps = [np.sort(rng.choice(n, k, replace=False)) for _ in range(40)]
    pool, counter = oracle.LruSlots(P), oracle.LruPool(P)
    for ids, (src, vict, inst, tags, last) in zip(steps, lru_slots_brute(steps, P, n)):
        plan = pool.plan(ids, n)
        assert plan.src_map.tolist() == src
        assert plan.victim.tolist() == vict and plan.install.tolist() == inst
        assert pool.tags == tags and pool.last_use == last
        assert int(np.sum(plan.src_map >= 0)) == counter.step(ids)
        # invariants: a token sits in one slot; every installed miss is resident
        resident = [t for t in pool.tags if t >= 0]
        assert len(resident) == len(set(resident))
        for t, keep in zip(plan.miss_ids, plan.install):
            assert (int(t) in resident) == bool(keep) or not keep


def test_lru_slots_hand_worked():
    pool = oracle.LruSlots(3)
    p = pool.plan([5, 9], 20)                 # cold: empty slots 0, 1
    assert p.victim.tolist() == [0, 1] and pool.tags == [5, 9, -1]
    p = pool.plan([1, 9], 20)                 # 9 hits (touched), 1 takes empty slot 2
    assert p.src_map.tolist() == [-2, 1] and p.victim.tolist() == [2]
    p = pool.plan([3], 20)                    # LRU is slot 0 (token 5, time 1)
    assert p.victim.tolist() == [0] and pool.tags == [3, 9, 1]
    assert pool.clock == 5 and pool.last_use == [5, 3, 4]
