"""Host-side legs of bench.py that need no GPU: the CPU baseline (the oracle on
one core and on every core, in worker processes) and the plan check that
follows a few requests through the bench's own forward input stream."""
import numpy as np

import bench
import oracle
import workload as wl


def test_cpu_baseline_leg_reports_one_core_and_all_cores():
    args = bench.parse(["--workload", "tiny", "--cpu-seconds", "0.2"])
    cb = bench.cpu_baseline_leg(args, wl.TINY, {})
    assert cb["kind"] == "oracle" and cb["unit"] == bench.UNIT
    assert cb["value"] > 0 and cb["single_core_value"] > 0
    assert cb["cores"] == 1            # tiny has one request: one worker
    assert cb["host_cores"] >= 1 and cb["cpu_model"] and cb["sample"]


def test_oracle_worker_rows_and_timing():
    out = bench.oracle_worker({"workload": "decode_batch", "overrides": {"B": 2, "H": 16},
                               "requests": [0, 1], "budget_s": 0.0})
    # the budget is spent after the first request's step
    assert out["requests"] == 1 and out["rows"] == 4 * 2048 and out["secs"] > 0


def _oracle_misses(w, steps, requests):
    lens = wl.ctx_lens(w)
    miss = np.zeros((steps.shape[0], w.B), np.int32)
    for b in requests:
        st = oracle.init_state(1, w.S, w.W)
        for t in range(steps.shape[0]):
            ids = oracle.topk_ids(steps[t, b], int(lens[b]), w.k)
            plan = oracle.dsa_plan(ids, int(lens[b]), st.tags, st.fifo_ptr, w.S, w.W)
            oracle.metadata_update(st.tags, st.fifo_ptr, plan)
            miss[t, b] = plan.miss_count
    return miss


def test_plan_check_agrees_with_a_matching_log_and_not_with_a_wrong_one():
    w = wl.scaled(wl.DECODE_BATCH, B=2, ctx=8192)
    stream = wl.ScoreStream(w)
    steps = np.stack([stream.next() for _ in range(6)])
    miss = _oracle_misses(w, steps, [0, 1])
    first, timed = 2, 4
    lens = wl.ctx_lens(w)
    r = bench.oracle_hit_check(w, steps, lens, first, timed, miss[first:first + timed], [0, 1])
    assert r["oracle_hit_rate"] == r["device_hit_rate"]
    assert 0.0 < r["oracle_hit_rate"] < 1.0
    bad = miss[first:first + timed].copy()
    bad[1, 0] += 1
    r = bench.oracle_hit_check(w, steps, lens, first, timed, bad, [0, 1])
    assert r["oracle_hit_rate"] != r["device_hit_rate"]
