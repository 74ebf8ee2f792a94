"""The fused serve-and-attend path (staged layout): the attention reads its
rows straight from the pool by the plan, with only the missed rows staged in
the pool tensor's extra rows (P + position). Checked through the C ABI:

* dsa_stage_misses: the staged rows are the host rows of the misses' first
  positions, bit for bit, and code-1 installs land in their victim slots;
* sfa_mla_decode_pool: bit-exact against sfa_mla_decode over the selection
  those rows make (same tiles, same arithmetic), including repeated tokens,
  ragged k and head counts that are not a multiple of 128; and within the
  attention tolerance of the float64 oracle;
* dsa_refill_pool_staged: the pool after the refill equals the oracle's;
* whole steps (layout "staged") against the oracle step by step."""
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


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _synthetic_plan(rng, B, k, P, hit_frac, repeats):
    """src_map with hits (slots) and misses (-1 - t), the ascending miss list
    with first positions, and the selection each position reads from a pool
    tensor of P + k rows per request."""
    src = np.empty((B, k), np.int32)
    mids = np.zeros((B, k), np.int32)
    mpos = np.zeros((B, k), np.int32)
    mcnt = np.zeros(B, np.int32)
    mrows = np.zeros(B, np.int32)
    row_of = np.empty((B, k), np.int64)
    for b in range(B):
        first = {}
        for j in range(k):
            if rng.random() < hit_frac:
                src[b, j] = rng.integers(0, P)
                row_of[b, j] = src[b, j]
                continue
            if repeats and first and rng.random() < 0.3:
                t = int(rng.choice(list(first)))
            else:
                t = int(rng.integers(0, 1 << 20))
                while t in first:
                    t = int(rng.integers(0, 1 << 20))
            first.setdefault(t, j)
            src[b, j] = -1 - t
            row_of[b, j] = P + first[t]
        ts = sorted(first)
        mcnt[b] = len(ts)
        mids[b, :len(ts)] = ts
        mpos[b, :len(ts)] = [first[t] for t in ts]
        mrows[b] = int(np.sum(src[b] < 0))
    return src, mids, mpos, mcnt, mrows, row_of


@pytest.mark.parametrize("B,H,k,repeats", [(2, 128, 2048, False), (3, 128, 300, False),
                                           (1, 16, 256, False), (2, 20, 513, True),
                                           (1, 128, 1, False), (2, 128, 1279, False),
                                           (1, 256, 1000, True), (4, 128, 4096, False)])
def test_sfa_pool_equals_selection_attention(d, B, H, k, repeats):
    rng = np.random.default_rng(B * 7 + H + k)
    P = 1024
    pool = wl.normal_bf16(B * (P + k), 576, 101, 9, k, H).reshape(B, P + k, 576)
    q = wl.normal_bf16(B * H, 576, 102, 9, k, H).reshape(B, H, 576)
    src, mids, mpos, mcnt, mrows, row_of = _synthetic_plan(rng, B, k, P, 0.7, repeats)
    if repeats:
        assert (mrows > mcnt).any()
    sel = np.stack([pool[b, row_of[b]] for b in range(B)])
    scale = 1 / math.sqrt(576)
    nbytes = d.sfa_workspace_size(B, H, k)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out_p = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    lse_p = torch.empty((B, H), dtype=torch.float32, device="cuda")
    out_s = torch.empty_like(out_p)
    lse_s = torch.empty_like(lse_p)
    err = _err()
    qt = _t(q.view(np.int16))
    assert d.sfa_mla_decode_pool(qt, _t(pool.view(np.int16)), P, _t(src), _t(mids), _t(mpos),
                                 _t(mcnt), _t(mrows), B, H, k, scale, out_p, lse_p, ws, nbytes,
                                 err) == 0
    assert d.ts_read_error(err) == 0
    assert d.sfa_mla_decode(qt, _t(sel.view(np.int16)), B, H, k, scale, out_s, lse_s, ws, nbytes,
                            err) == 0
    assert d.ts_read_error(err) == 0
    assert torch.equal(out_p.view(torch.int16), out_s.view(torch.int16))
    assert torch.equal(lse_p, lse_s)
    got = out_p.cpu().view(torch.int16).numpy().view(np.uint16)
    o, _ = oracle.sfa_decode(q[0], sel[0], scale)
    a, rel = sfa_errors(got[0], oracle.round_to_bf16_bits(o))
    assert a <= SFA_ABS_TOL and rel <= SFA_MEAN_REL_TOL, (a, rel)


def test_sfa_pool_flags_bad_slots(d):
    B, H, k, P = 1, 128, 64, 32
    pool = torch.zeros((B, P + k, 576), dtype=torch.int16, device="cuda")
    q = torch.zeros((B, H, 576), dtype=torch.int16, device="cuda")
    src = torch.zeros((B, k), dtype=torch.int32, device="cuda")
    src[0, 3] = P + 5                           # a slot past the pool
    src[0, 4] = -(1 << 31)                      # an invalid id
    mids = torch.zeros((B, k), dtype=torch.int32, device="cuda")
    mcnt = torch.zeros((B,), dtype=torch.int32, device="cuda")
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    nbytes = d.sfa_workspace_size(B, H, k)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    err = _err()
    assert d.sfa_mla_decode_pool(q, pool, P, src, mids, mids, mcnt, mcnt, B, H, k, 0.1, out, None,
                                 ws, nbytes, err) == 0
    bits = d.ts_read_error(err)
    assert bits & 0x04 and bits & 0x01


def test_stage_misses_and_staged_refill(d):
    from decode_dsa_kv_gb300 import HostKV
    rng = np.random.default_rng(14)
    B, S, W, k, ctx = 3, 64, 4, 300, 3000
    P = S * W
    host = HostKV(1, B, ctx)
    host.array[...] = rng.integers(0, 65536, size=host.array.shape, dtype=np.uint16)
    lens = np.array([ctx, 2000, 1500], np.int32)
    tags = np.full((B, P), -1, np.int32)
    ptr = rng.integers(0, W, size=(B, S)).astype(np.int32)
    for b in range(B):                       # a partly filled pool holding its tagged rows
        for st in range(S):
            cand = rng.choice(np.arange(st, int(lens[b]), S), W, replace=False)
            for w_ in range(W):
                if rng.random() < 0.8:
                    tags[b, st * W + w_] = cand[w_]
    pool = rng.integers(0, 65536, size=(B, P + k, 576), dtype=np.uint16)
    for b in range(B):
        for slot in np.flatnonzero(tags[b] >= 0):
            pool[b, slot] = host.array[0, b, tags[b, slot]]
    ids = np.stack([np.sort(rng.choice(int(n), k, replace=False)) for n in lens]).astype(np.int32)
    i32 = dict(dtype=torch.int32, device="cuda")
    out = {n: torch.empty((B, k), **i32) for n in ("src_map", "miss_ids", "miss_pos", "victim")}
    install = torch.empty((B, k), dtype=torch.uint8, device="cuda")
    mcnt = torch.empty((B,), **i32)
    mrows = torch.empty((B,), **i32)
    pnext = torch.empty((B, S), **i32)
    err = _err()
    ln = _t(lens)
    tags_t, ptr_t = _t(tags), _t(ptr)
    assert d.dsa_plan(_t(ids), ln, B, k, tags_t, ptr_t, S, W, out["src_map"], out["miss_ids"],
                      out["miss_pos"], out["victim"], install, mcnt, mrows, pnext, err) == 0
    pool_t = _t(pool.view(np.int16))
    assert d.dsa_stage_misses(out["miss_ids"], out["miss_pos"], mcnt, out["victim"], install, B, k,
                              pool_t, P, host.layer_ptr(0), ctx, ln, err) == 0
    assert d.ts_read_error(err) == 0
    staged = pool_t.cpu().numpy().view(np.uint16)
    mid = out["miss_ids"].cpu().numpy()
    mps = out["miss_pos"].cpu().numpy()
    vic = out["victim"].cpu().numpy()
    ins = install.cpu().numpy()
    for b in range(B):
        M = int(mcnt[b])
        plan = oracle.dsa_plan(ids[b], int(lens[b]), tags[b], ptr[b], S, W)
        assert np.array_equal(mid[b, :M], plan.miss_ids)
        codes = plan.install_code
        for i in range(M):
            assert np.array_equal(staged[b, P + mps[b, i]], host.array[0, b, mid[b, i]])
            if codes[i] == 1:                # written on arrival
                assert np.array_equal(staged[b, vic[b, i]], host.array[0, b, mid[b, i]])
        assert np.array_equal(ins[b, :M], codes)
    # the refill from the staging rows, with the metadata update
    assert d.dsa_refill_pool_staged(out["miss_ids"], out["miss_pos"], out["victim"], install,
                                    mcnt, B, k, pool_t, P, 1, tags_t, ptr_t, pnext, S, W,
                                    err) == 0
    assert d.ts_read_error(err) == 0
    after = pool_t.cpu().numpy().view(np.uint16)
    for b in range(B):
        plan = oracle.dsa_plan(ids[b], int(lens[b]), tags[b], ptr[b], S, W)
        pb = pool[b, :P].copy()
        oracle.dsa_install(pb, plan, host.array[0, b])
        tb, qb = tags[b].copy(), ptr[b].copy()
        oracle.metadata_update(tb, qb, plan)
        assert np.array_equal(after[b, :P], pb)
        assert np.array_equal(tags_t[b].cpu().numpy(), tb)
        assert np.array_equal(ptr_t[b].cpu().numpy(), qb)
    host.close()


def run_staged_steps(d, w, steps, sample=None, sfa_layers=None, sfa_heads=None):
    """Whole steps with the staged layout against the oracle, per step: ids,
    plan, staged rows and the pool after the step bit-exact; each checked
    layer's attention bit-exact against sfa_mla_decode over the oracle's
    selection and within tolerance of the float64 oracle."""
    lens = wl.ctx_lens(w)
    host = d.HostKV(w.layers, w.B, w.ctx_stride)
    wl.fill_host_kv(w, host.array)
    g = d.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host,
                      layout="staged")
    sample = list(range(w.B)) if sample is None else sample
    sfa_layers = list(range(w.layers)) if sfa_layers is None else sfa_layers
    heads = slice(None) if sfa_heads is None else sfa_heads
    states = {b: oracle.init_state(w.layers, w.S, w.W) for b in sample}
    stream = wl.ScoreStream(w)
    scale = 1 / math.sqrt(576)
    P = w.P
    ws_bytes = d.sfa_workspace_size(1, w.H, w.k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    err = _err()
    rates = []
    for step in range(steps):
        scores = stream.next()
        q = wl.queries(w, step)
        g.step(torch.from_numpy(scores).cuda(), torch.from_numpy(q.view(np.int16)).cuda())
        assert g.synchronize() == 0, f"device error bits at step {step}"
        ids = g.ids.cpu().numpy()
        src = g.src_map.cpu().numpy()
        rates.append(float((src >= 0).mean()))
        for b in sample:
            r = oracle.decode_step(states[b], scores[b], int(lens[b]), w.k, w.S, w.W,
                                   host.array[:, b], q[:, b], scale, with_sfa=False)
            plan = r["plan"]
            M = plan.miss_count
            assert np.array_equal(ids[b], r["ids"]), (step, b)
            assert np.array_equal(src[b], plan.src_map), (step, b)
            assert int(g.miss_count[b]) == M
            assert np.array_equal(g.install[b, :M].cpu().numpy(), plan.install_code)
            assert np.array_equal(g.tags[b].cpu().numpy(), states[b].tags)
            assert np.array_equal(g.fifo_ptr[b].cpu().numpy(), states[b].fifo_ptr)
            for l in range(w.layers):
                pool = g.pool[l, b].cpu().numpy().view(np.uint16)
                assert np.array_equal(pool[:P], states[b].pool[l]), (step, b, l)
                assert np.array_equal(pool[P + plan.miss_pos], host.array[l, b][plan.miss_ids])
            for l in sfa_layers:
                out = torch.empty((1, w.H, 512), dtype=torch.bfloat16, device="cuda")
                qb = torch.from_numpy(np.ascontiguousarray(q[l, b:b + 1]).view(np.int16)).cuda()
                selb = torch.from_numpy(np.ascontiguousarray(r["sel"][l][None]).view(np.int16))
                assert d.sfa_mla_decode(qb, selb.cuda(), 1, w.H, w.k, scale, out, None, ws,
                                        ws_bytes, err) == 0
                assert d.ts_read_error(err) == 0
                assert torch.equal(g.out[l, b].view(torch.int16), out[0].view(torch.int16)), \
                    (step, b, l)
                o, _ = oracle.sfa_decode(q[l, b][heads], r["sel"][l], scale)
                got = g.out[l, b].cpu().view(torch.int16).numpy().view(np.uint16)[heads]
                a, rel = sfa_errors(got, oracle.round_to_bf16_bits(o))
                assert a <= SFA_ABS_TOL and rel <= SFA_MEAN_REL_TOL, (step, b, l, a, rel)
    host.close()
    return rates


def test_staged_tiny_all_steps(d):
    rates = run_staged_steps(d, wl.TINY, wl.TINY.steps)
    assert rates[0] == 0.0 and max(rates[1:]) > 0.3


def test_staged_decode_batch_scaled(d):
    rates = run_staged_steps(d, wl.scaled(wl.DECODE_BATCH, B=3, ctx=16384, S=256), 5,
                             sfa_layers=[0, 3])
    assert rates[-1] > 0.3


def test_staged_long_context_scaled(d):
    run_staged_steps(d, wl.scaled(wl.LONG_CONTEXT, B=2), 4, sfa_layers=[1])


def test_staged_adversarial_full_size(d):
    # 4 x 1,048,576 positions (19 GB of host KV, the wide miss grid) with the
    # overflowing request; the oracle follows requests 0 and 3
    run_staged_steps(d, wl.ADVERSARIAL, 2, sample=[0, 3], sfa_layers=[3],
                     sfa_heads=slice(0, 128, 11))


def test_staged_large_batch_full_size(d):
    rates = run_staged_steps(d, wl.LARGE_BATCH, 5, sample=[0, 127], sfa_layers=[2],
                             sfa_heads=slice(0, 128, 13))
    assert rates[0] == 0.0 and rates[-1] > 0.3


def test_staged_decode_batch_full_size(d):
    run_staged_steps(d, wl.DECODE_BATCH, 3, sample=[0, 31], sfa_layers=[0, 3],
                     sfa_heads=slice(0, 128, 9))


@pytest.mark.parametrize("w,steps", [(wl.LARGE_BATCH, 6), (wl.DECODE_BATCH, 4)])
def test_streamed_attention_equals_layer_waits(d, w, steps):
    """Streamed attention (each CTA waits inside the kernel for its own
    request's staged rows while the gather still runs) against attention that
    waits for the whole layer: the same outputs and pool, bit for bit, step
    after step at full size (the streamed group is the one the whole-step
    tests above check against the oracle)."""
    lens = wl.ctx_lens(w)
    host = d.HostKV(w.layers, w.B, w.ctx_stride)
    wl.fill_host_kv(w, host.array)
    gs = [d.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host,
                        layout="staged", streamed=s) for s in (True, False)]
    assert gs[0].arrived is not None and gs[1].arrived is None
    stream = wl.ScoreStream(w)
    for step in range(steps):
        scores = torch.from_numpy(stream.next()).cuda()
        q = torch.from_numpy(wl.queries(w, step).view(np.int16)).cuda()
        for g in gs:
            g.step(scores, q)
        for g in gs:
            assert g.synchronize() == 0, step
        assert torch.equal(gs[0].out.view(torch.int16), gs[1].out.view(torch.int16)), step
        assert torch.equal(gs[0].src_map, gs[1].src_map), step
        for l in range(w.layers):
            assert torch.equal(gs[0].pool[l], gs[1].pool[l]), (step, l)
        # every layer's arrival counts reached the requests' miss counts
        arr = gs[0].arrived[:w.layers * w.B].view(w.layers, w.B)
        assert torch.equal(arr, gs[0].miss_count[None].expand(w.layers, -1)), step
    host.close()
