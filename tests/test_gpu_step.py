"""Whole decode steps through the per-step schedule (top-k, one plan per group,
per-layer gather and SFA, then the refill of every layer with the metadata
update on the side stream), compared with the oracle run step by step on the
same seeded inputs: bit-exact ids, plan, selection bytes and pool state; SFA
within tolerance."""
import math

import numpy as np
import pytest

import oracle
import workload as wl
from _util import SFA_ABS_TOL, SFA_MEAN_REL_TOL, ensure_library, sfa_errors

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def d():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()
    import decode_dsa_kv_gb300 as d
    return d


def run_steps(d, w, steps, sample=None, sfa_layers=None, sfa_heads=None):
    """Run `steps` decode steps of workload `w` on the GPU and, for the
    requests in `sample` (default: all), on the oracle; compare after each
    step. Returns per-step hit rates of the GPU plan and the number of
    installs whose victim slot was read as a hit in the same step (install
    code 2: the refill writes them after the layer's reads; the gather writes
    the others on arrival)."""
    lens = wl.ctx_lens(w)
    host = d.HostKV(w.layers, w.B, w.ctx_stride)
    wl.fill_host_kv(w, host.array)
    g = d.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host)
    sample = list(range(w.B)) if sample is None else sample
    sfa_layers = list(range(w.layers)) if sfa_layers is None else sfa_layers
    states = {b: oracle.init_state(w.layers, w.S, w.W) for b in sample}
    scores_stream = wl.ScoreStream(w)
    scale = 1 / math.sqrt(576)
    hit_rates = []
    deferred = 0
    for step in range(steps):
        scores = scores_stream.next()
        q = wl.queries(w, step)
        g.step(torch.from_numpy(scores).cuda(), torch.from_numpy(q.view(np.int16)).cuda())
        assert g.synchronize() == 0, f"device error bits at step {step}"
        ids = g.ids.cpu().numpy()
        src = g.src_map.cpu().numpy()
        mc = g.miss_count.cpu().numpy()
        hit_rates.append(float((src >= 0).mean()))
        for b in sample:
            r = oracle.decode_step(states[b], scores[b], int(lens[b]), w.k, w.S, w.W,
                                   host.array[:, b], q[:, b], scale, with_sfa=False)
            plan = r["plan"]
            M = plan.miss_count
            assert np.array_equal(ids[b], r["ids"]), (step, b)
            assert np.array_equal(src[b], plan.src_map), (step, b)
            assert mc[b] == M
            assert int(g.miss_rows[b]) == plan.miss_rows
            assert np.array_equal(g.miss_ids[b, :M].cpu().numpy(), plan.miss_ids)
            assert np.array_equal(g.victim[b, :M].cpu().numpy(), plan.victim)
            assert np.array_equal(g.install[b, :M].cpu().numpy(), plan.install_code)
            deferred += int(np.sum(plan.install_code == 2))
            assert np.array_equal(g.tags[b].cpu().numpy(), states[b].tags), (step, b)
            assert np.array_equal(g.fifo_ptr[b].cpu().numpy(), states[b].fifo_ptr)
            for l in range(w.layers):
                sel = g.sel[l, b].cpu().numpy().view(np.uint16)
                assert np.array_equal(sel, r["sel"][l]), (step, b, l)
                assert np.array_equal(g.pool[l, b].cpu().numpy().view(np.uint16),
                                      states[b].pool[l]), (step, b, l)
            for l in sfa_layers:
                heads = slice(None) if sfa_heads is None else sfa_heads
                o, _ = oracle.sfa_decode(q[l, b][heads], r["sel"][l], scale)
                got = g.out[l, b].cpu().view(torch.int16).numpy().view(np.uint16)[heads]
                a, rel = sfa_errors(got, oracle.round_to_bf16_bits(o))
                assert a <= SFA_ABS_TOL and rel <= SFA_MEAN_REL_TOL, (step, b, l, a, rel)
    host.close()
    return hit_rates, deferred


def run_steps_reuse(d, w, steps, sfa_layers=(0,)):
    """Decode steps with the adjacent-step reuse policy, against the oracle's
    plan_reuse step by step: bit-exact ids, plan and selection bytes (which
    must equal the host rows of the ids), SFA within tolerance. Returns the
    per-step hit rates."""
    lens = wl.ctx_lens(w)
    host = d.HostKV(w.layers, w.B, w.ctx_stride)
    wl.fill_host_kv(w, host.array)
    g = d.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host, policy="reuse")
    prev = {b: np.full(w.k, -1, np.int32) for b in range(w.B)}
    scores_stream = wl.ScoreStream(w)
    scale = 1 / math.sqrt(576)
    rates = []
    for step in range(steps):
        scores = scores_stream.next()
        q = wl.queries(w, step)
        g.step(torch.from_numpy(scores).cuda(), torch.from_numpy(q.view(np.int16)).cuda())
        assert g.synchronize() == 0, f"device error bits at step {step}"
        ids = g.ids.cpu().numpy()
        src = g.src_map.cpu().numpy()
        rates.append(float((src >= 0).mean()))
        for b in range(w.B):
            ref_ids = oracle.topk_ids(scores[b], int(lens[b]), w.k)
            assert np.array_equal(ids[b], ref_ids), (step, b)
            p = oracle.plan_reuse(ref_ids, prev[b], int(lens[b]))
            assert np.array_equal(src[b], p.src_map), (step, b)
            M = p.miss_count
            assert int(g.miss_count[b]) == M and int(g.miss_rows[b]) == M
            assert np.array_equal(g.miss_ids[b, :M].cpu().numpy(), p.miss_ids)
            assert np.array_equal(g.miss_pos[b, :M].cpu().numpy(), p.miss_pos)
            for l in range(w.layers):
                sel = g.sel[l, b].cpu().numpy().view(np.uint16)
                assert np.array_equal(sel, host.array[l, b, ref_ids]), (step, b, l)
            for l in sfa_layers:
                o, _ = oracle.sfa_decode(q[l, b], host.array[l, b, ref_ids], scale)
                got = g.out[l, b].cpu().view(torch.int16).numpy().view(np.uint16)
                a_err, rel = sfa_errors(got, oracle.round_to_bf16_bits(o))
                assert a_err <= SFA_ABS_TOL and rel <= SFA_MEAN_REL_TOL, (step, b, l, a_err, rel)
            prev[b] = ref_ids
    host.close()
    return rates


def test_reuse_policy_tiny(d):
    rates = run_steps_reuse(d, wl.TINY, wl.TINY.steps)
    assert rates[0] == 0.0 and max(rates[1:]) > 0.3


def test_reuse_policy_decode_batch_scaled(d):
    # the base design's reuse hits less often than the 8192-entry FIFO pool on
    # the same score process (it keeps only the previous selection)
    w = wl.scaled(wl.DECODE_BATCH, B=2)
    reuse = run_steps_reuse(d, w, 5, sfa_layers=(2,))
    fifo, _ = run_steps(d, w, 5, sfa_layers=[])
    assert 0.45 < np.mean(reuse[1:]) < 0.75
    assert np.mean(fifo[1:]) > np.mean(reuse[1:])


def test_tiny_all_steps(d):
    rates, _ = run_steps(d, wl.TINY, wl.TINY.steps)
    assert rates[0] == 0.0 and max(rates[1:]) > 0.3


def test_decode_batch_scaled(d):
    w = wl.scaled(wl.DECODE_BATCH, B=3)
    rates, deferred = run_steps(d, w, 5, sfa_layers=[0, 3])
    assert rates[-1] > 0.5
    assert deferred > 0  # both install paths ran


def test_long_context_scaled(d):
    w = wl.scaled(wl.LONG_CONTEXT, B=2)
    run_steps(d, w, 4, sfa_layers=[1])


def test_adversarial_scaled_overflow(d):
    w = wl.scaled(wl.ADVERSARIAL, ctx=1 << 17)
    run_steps(d, w, 3, sfa_layers=[2])


def test_decode_batch_mtp_folded_queries(d):
    # MTP reuse: two draft steps share the step's selection; their queries are
    # folded into the heads (3 x 128), as the group step runs them
    w = wl.scaled(wl.DECODE_BATCH, B=2, H=3 * 128)
    run_steps(d, w, 2, sfa_layers=[1], sfa_heads=slice(0, 384, 7))


def test_decode_batch_full_size_sampled(d):
    # the full workload (32 requests x 65,536 tokens x 4 layers) in the bench's
    # launch configuration; the oracle follows four of the requests
    w = wl.DECODE_BATCH
    run_steps(d, w, 3, sample=[0, 13, 31], sfa_layers=[0, 3], sfa_heads=slice(0, 128, 9))


def test_large_batch_scaled(d):
    # the large-batch shape (128 requests, 8192-entry pools, 128 heads: the
    # plan, gather and attention grids at their widest) with contexts cut to
    # 16,384 positions (32 tokens per set, so sets fill and evict); the oracle
    # follows four requests
    w = wl.scaled(wl.LARGE_BATCH, ctx=16384)
    rates, _ = run_steps(d, w, 4, sample=[0, 57, 100, 127], sfa_layers=[2],
                         sfa_heads=slice(0, 128, 5))
    assert rates[0] == 0.0 and rates[-1] > 0.4


def test_adversarial_full_size_sampled(d):
    # the full adversarial workload (4 requests x 1,048,576 positions, 19 GB of
    # host KV): the bench's launch configuration, including the gather's grid
    # for host KV over 12 GB; the oracle follows requests 0 and 3 (the
    # overflowing one)
    w = wl.ADVERSARIAL
    rates, _ = run_steps(d, w, 2, sample=[0, 3], sfa_layers=[3], sfa_heads=slice(0, 128, 11))
    assert max(rates) < 0.2


def test_large_batch_full_size_sampled(d):
    # the full large-batch workload (128 requests x 32,768 positions x 4 layers,
    # 19 GB of host KV), the bench's default configuration and launch grid; the
    # oracle follows the first and the last request
    w = wl.LARGE_BATCH
    rates, _ = run_steps(d, w, 5, sample=[0, 127], sfa_layers=[1], sfa_heads=slice(0, 128, 13))
    assert rates[0] == 0.0 and rates[-1] > 0.3
