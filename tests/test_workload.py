"""The seeded synthetic workloads: sizes match the page's constants, the score
processes have the statistics they are meant to have, the generator is
deterministic row by row."""
import json
import os

import numpy as np

import workload as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pool_constants.json")


def test_sizes_follow_the_page():
    g = json.load(open(GOLDEN))
    for w in wl.WORKLOADS[1:]:
        assert w.k == g["topk"]
        assert w.layers == g["group_layers"]
        assert w.W == g["set_associativity"]
        assert w.P in (g["default_pool_size"], g["large_pool_size"])
        assert w.P // g["set_associativity"] == w.S     # one counter per set
    assert wl.LONG_CONTEXT.P == g["large_pool_size"]
    assert wl.DECODE_BATCH.P == g["default_pool_size"]
    for w in wl.WORKLOADS[1:4]:
        assert w.overlap == g["adjacent_step_reuse"]


def test_generator_rows_are_deterministic_and_normal():
    a = wl.normal_bf16(2000, 576, 99, 1, 2, 3)
    b = wl.normal_bf16(1, 576, 99, 1, 2, 3, row0=1234)
    assert np.array_equal(a[1234], b[0])
    f = wl.bf16_to_f32(a).astype(np.float64)
    assert abs(f.mean()) < 0.01 and abs(f.std() - 1) < 0.01
    c = wl.normal_bf16(10, 576, 99, 1, 2, 4)
    assert not np.array_equal(a[:10], c)


def _overlap(prev, cur, k, n):
    a = set(np.argpartition(-prev[:n], k)[:k].tolist())
    b = set(np.argpartition(-cur[:n], k)[:k].tolist())
    return len(a & b) / k


def test_ar1_overlap_near_target():
    w = wl.scaled(wl.DECODE_BATCH, B=3)
    st = wl.ScoreStream(w)
    prev = st.next()
    ovs = []
    for _ in range(5):
        cur = st.next()
        for b in range(w.B):
            ovs.append(_overlap(prev[b], cur[b], w.k, w.ctx))
        prev = cur
    assert abs(np.mean(ovs) - 0.60) < 0.04, np.mean(ovs)


def test_long_context_lengths_and_hot_set():
    w = wl.LONG_CONTEXT
    lens = wl.ctx_lens(w)
    assert lens.min() >= 30000 and lens.max() <= 200000 and len(set(lens.tolist())) > 1
    st = wl.ScoreStream(wl.scaled(w, B=2))
    s = st.next()
    assert np.isnan(s[0, lens[0]:]).all() and not np.isnan(s[0, :lens[0]]).any()


def test_adversarial_ties_and_set_flood():
    w = wl.scaled(wl.ADVERSARIAL, ctx=1 << 17)
    st = wl.ScoreStream(w)
    s = st.next()
    b = w.overflow_request
    top = np.argpartition(-s[b], w.k)[:w.k]
    assert int(np.sum(top % w.S == w.overflow_set)) >= w.overflow_count
    # exact repeats of grid values among the scores
    vals, counts = np.unique(s[0], return_counts=True)
    assert counts.max() > 10
