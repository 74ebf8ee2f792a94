"""Invariants of the oracle's whole decode step (GLM-5.2 shared-Indexer KV Cache
Offload page: §4.1 groups, §4.2 one plan per group, §4.3 FIFO pool, §4.4 SFA
first and refill later, §5.1 metadata update at the group's last layer)."""
import math

import numpy as np

import workload as wl
from oracle import decode_step, init_state


def _check_state(state, host, S, W, layers):
    for s in range(S):
        held = [t for t in state.tags[s * W:(s + 1) * W] if t >= 0]
        assert len(held) == len(set(held)) and all(t % S == s for t in held)
    assert np.all((state.fifo_ptr >= 0) & (state.fifo_ptr < W))
    for slot, t in enumerate(state.tags):
        if t >= 0:
            for l in range(layers):
                assert np.array_equal(state.pool[l][slot], host[l][t])


def test_tiny_workload_steps():
    w = wl.TINY
    lens = wl.ctx_lens(w)
    host = np.zeros((w.layers, w.B, w.ctx_stride, 576), np.uint16)
    wl.fill_host_kv(w, host)
    stream = wl.ScoreStream(w)
    state = init_state(w.layers, w.S, w.W)
    hit_rates = []
    for step in range(w.steps):
        scores = stream.next()
        q = wl.queries(w, step)
        r = decode_step(state, scores[0], int(lens[0]), w.k, w.S, w.W,
                        host[:, 0], q[:, 0], 1 / math.sqrt(576))
        plan = r["plan"]
        hits = int((plan.src_map >= 0).sum())
        assert hits + plan.miss_count == w.k
        hit_rates.append(hits / w.k)
        # every served row, hit or miss, is the host row of its token: a hit's
        # slot was read before this step's refill could overwrite it
        for l in range(w.layers):
            assert np.array_equal(r["sel"][l], host[l, 0][r["ids"]])
            assert r["out"][l].shape == (w.H, 512)
        _check_state(state, host[:, 0], w.S, w.W, w.layers)
    assert hit_rates[0] == 0.0              # cold pool
    assert max(hit_rates[1:]) > 0.3          # the walk keeps many positions


def test_repeat_step_is_all_hits_without_overflow():
    S, W, ctx, k = 8, 2, 64, 8
    host = [np.arange(ctx * 576, dtype=np.uint16).reshape(ctx, 576)]
    q = [np.zeros((2, 576), np.uint16)]
    scores = np.zeros(ctx, np.float32)
    scores[8:16] = 5.0                      # ids 8..15: one per set
    state = init_state(1, S, W)
    r1 = decode_step(state, scores, ctx, k, S, W, host, q, 0.1)
    assert r1["plan"].miss_count == k
    r2 = decode_step(state, scores, ctx, k, S, W, host, q, 0.1)
    assert r2["plan"].miss_count == 0 and np.all(r2["plan"].src_map >= 0)
    assert state.fifo_ptr.tolist() == [1] * S   # hits did not move the pointers
