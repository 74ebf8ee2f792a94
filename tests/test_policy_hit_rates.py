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
