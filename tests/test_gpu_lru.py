"""The fully associative LRU pool on the device (dsa_plan_lru and the group
step's LRU policy; GLM-5.2 shared-Indexer KV Cache Offload, §3, the pool the
pages measured before the set-associative FIFO of §4.3), against the oracle's
slot-level LRU pool (oracle.LruSlots): bit-exact source maps, miss lists,
victims, install flags, tags and the slots' recency order (the oracle's slots
sorted by empty first, then last use, then index), step after step; and whole
decode steps (both layouts) with the pool's rows."""
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


@pytest.mark.parametrize("B,P,k,ctx,steps", [(3, 1024, 256, 4000, 14), (2, 600, 300, 1500, 10),
                                             (1, 8192, 2048, 65536, 6)])
def test_plan_lru_matches_oracle_step_by_step(d, B, P, k, ctx, steps):
    rng = np.random.default_rng(P + k)
    i32 = dict(dtype=torch.int32, device="cuda")
    tags = torch.full((B, P), -1, **i32)
    order = torch.arange(P, **i32).repeat(B, 1)
    out = {n: torch.empty((B, k), **i32) for n in ("src", "mids", "mpos", "victim")}
    install = torch.empty((B, k), dtype=torch.uint8, device="cuda")
    mcnt = torch.empty((B,), **i32)
    mrows = torch.empty((B,), **i32)
    err = torch.zeros(1, **i32)
    lens = torch.full((B,), ctx, **i32)
    pools = [oracle.LruSlots(P) for _ in range(B)]
    # a slowly moving selection, so that hits, evictions and empty slots mix
    base = [np.sort(rng.choice(ctx, k, replace=False)) for _ in range(B)]
    for step in range(steps):
        ids = np.empty((B, k), np.int32)
        for b in range(B):
            keep = base[b][rng.random(k) < 0.6]
            new = rng.choice(np.setdiff1d(np.arange(ctx), keep), k - keep.size, replace=False)
            base[b] = np.sort(np.concatenate([keep, new]))
            ids[b] = base[b]
        assert d.dsa_plan_lru(torch.from_numpy(ids).cuda(), lens, B, k, tags, order, P,
                              out["src"], out["mids"], out["mpos"], out["victim"], install, mcnt,
                              mrows, err) == 0
        assert d.ts_read_error(err) == 0
        for b in range(B):
            plan = pools[b].plan(ids[b], ctx)
            M = plan.miss_count
            assert np.array_equal(out["src"][b].cpu().numpy(), plan.src_map), (step, b)
            assert int(mcnt[b]) == M and int(mrows[b]) == M
            assert np.array_equal(out["mids"][b, :M].cpu().numpy(), plan.miss_ids)
            assert np.array_equal(out["mpos"][b, :M].cpu().numpy(), plan.miss_pos)
            assert np.array_equal(out["victim"][b, :M].cpu().numpy(), plan.victim), (step, b)
            assert np.array_equal(install[b, :M].cpu().numpy(), plan.install_code)
            assert np.array_equal(tags[b].cpu().numpy(), np.asarray(pools[b].tags))
            want = sorted(range(P), key=lambda s: (pools[b].tags[s] >= 0,
                                                   pools[b].last_use[s], s))
            assert np.array_equal(order[b].cpu().numpy(), want), (step, b)


def test_plan_lru_flags_unsorted_ids(d):
    i32 = dict(dtype=torch.int32, device="cuda")
    B, P, k = 1, 64, 4
    ids = torch.tensor([[5, 3, 9, 11]], **i32)
    z = lambda *s: torch.zeros(s, **i32)
    err = z(1)
    assert d.dsa_plan_lru(ids, torch.tensor([100], **i32), B, k, torch.full((B, P), -1, **i32),
                          torch.arange(P, **i32)[None], P, z(B, k), z(B, k), z(B, k), z(B, k),
                          torch.zeros((B, k), dtype=torch.uint8, device="cuda"), z(B), z(B),
                          err) == 0
    assert d.ts_read_error(err) & 0x80
    from decode_dsa_kv_gb300 import _abi
    # k above the pool size is refused on the host
    assert d.dsa_plan_lru(ids, torch.tensor([100], **i32), B, k, z(B, 2), z(B, 2), 2, z(B, k),
                          z(B, k), z(B, k), z(B, k),
                          torch.zeros((B, k), dtype=torch.uint8, device="cuda"), z(B), z(B),
                          err) == _abi.TS_ERR_UNSUPPORTED


@pytest.mark.parametrize("fault", ["order_repeats_a_slot", "order_out_of_range", "tag_twice"])
def test_plan_lru_flags_corrupt_metadata(d, fault):
    """A recency order that is not a permutation of the slots, or a token held
    by two slots, is reported; the plan installs nothing and leaves the order
    as it was."""
    i32 = dict(dtype=torch.int32, device="cuda")
    B, P, k = 1, 64, 4
    ids = torch.tensor([[3, 5, 9, 11]], **i32)
    tags = torch.full((B, P), -1, **i32)
    tags[0, 10] = 5
    order = torch.arange(P, **i32)[None].clone()
    if fault == "order_repeats_a_slot":
        order[0, 7] = 6
    elif fault == "order_out_of_range":
        order[0, 7] = P
    else:
        tags[0, 20] = 5
    before = order.clone()
    z = lambda *s: torch.zeros(s, **i32)
    victim = torch.full((B, k), 77, **i32)
    install = torch.ones((B, k), dtype=torch.uint8, device="cuda")
    err = z(1)
    mcnt = z(B)
    assert d.dsa_plan_lru(ids, torch.tensor([100], **i32), B, k, tags, order, P, z(B, k), z(B, k),
                          z(B, k), victim, install, mcnt, z(B), err) == 0
    assert d.ts_read_error(err) & 0x04
    assert torch.equal(order, before)
    M = int(mcnt[0])
    assert M == 3 and int(install[0, :M].sum()) == 0


@pytest.mark.parametrize("layout", ["selection", "staged"])
@pytest.mark.parametrize("w,steps,sample", [
    (wl.scaled(wl.TINY), 4, None),
    (wl.scaled(wl.DECODE_BATCH, B=2, ctx=16384, S=256), 6, None),
])
def test_lru_whole_steps(d, layout, w, steps, sample):
    lens = wl.ctx_lens(w)
    host = d.HostKV(w.layers, w.B, w.ctx_stride)
    wl.fill_host_kv(w, host.array)
    g = d.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host, policy="lru",
                      layout=layout)
    sample = list(range(w.B)) if sample is None else sample
    pools = {b: oracle.LruSlots(w.P) for b in sample}
    data = {b: np.zeros((w.layers, w.P, 576), np.uint16) for b in sample}
    stream = wl.ScoreStream(w)
    scale = 1 / math.sqrt(576)
    P = w.P
    rates = []
    for step in range(steps):
        scores = stream.next()
        q = wl.queries(w, step)
        g.step(torch.from_numpy(scores).cuda(), torch.from_numpy(q.view(np.int16)).cuda())
        assert g.synchronize() == 0, step
        src = g.src_map.cpu().numpy()
        rates.append(float((src >= 0).mean()))
        for b in sample:
            ids = oracle.topk_ids(scores[b], int(lens[b]), w.k)
            assert np.array_equal(g.ids[b].cpu().numpy(), ids)
            plan = pools[b].plan(ids, int(lens[b]))
            assert np.array_equal(src[b], plan.src_map), (step, b)
            assert np.array_equal(g.tags[b].cpu().numpy(), np.asarray(pools[b].tags))
            for l in range(w.layers):
                sel = oracle.dsa_serve(plan.src_map, data[b][l], host.array[l, b], int(lens[b]))
                assert np.array_equal(sel, host.array[l, b][ids])
                oracle.dsa_install(data[b][l], plan, host.array[l, b])
                pool = g.pool[l, b].cpu().numpy().view(np.uint16)
                assert np.array_equal(pool[:P], data[b][l]), (step, b, l)
                if layout == "selection":
                    assert np.array_equal(g.sel[l, b].cpu().numpy().view(np.uint16), sel)
                o, _ = oracle.sfa_decode(q[l, b], sel, scale)
                got = g.out[l, b].cpu().view(torch.int16).numpy().view(np.uint16)
                a, rel = sfa_errors(got, oracle.round_to_bf16_bits(o))
                assert a <= SFA_ABS_TOL and rel <= SFA_MEAN_REL_TOL, (step, b, l, a, rel)
    assert rates[0] == 0.0 and max(rates[1:]) > 0.3
    host.close()
