"""Failure and ordering paths on the GPU, in the forms that fault nothing.

* A bounded wait that runs out: with the attention's wait limit set to 1 ns,
  its waits give up at once; the call must report TS_DEVERR_TIMEOUT through the
  error word (no trap), let its copies land, free its tensor memory, and leave
  the next call, at the default limit, computing the right answer.
* Widened race windows in the group step: a spin kernel put on one of the
  three streams ahead of a step delays that stream's work by milliseconds.
  The step's cross-stream waits must still order every consumer after its
  producer: a plan after the previous step's refill (GLM-5.2 shared-Indexer KV
  Cache Offload, §4.4: each layer reads its rows before its refill; the next
  plan reads the tags the refill writes), a gather after its plan, the
  attention and the refill after the layer's gather. Every step is then
  compared with the oracle, bit for bit (ids, plan, selection, pool) and
  within tolerance (attention) - the hazard class of a read before the data is
  ready, which the GLM-5 serving post's HiCache fix is about."""
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


def _sfa(d, q, sel, B, H, k, scale):
    out = torch.zeros((B, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    nbytes = d.sfa_workspace_size(B, H, k)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert d.sfa_mla_decode(q, sel, B, H, k, scale, out, lse, ws, nbytes, err) == 0
    return out, d.ts_read_error(err)


@pytest.mark.parametrize("k", [2048, 1279])   # 4 chunks; 3 chunks, the last one ragged
def test_attention_wait_that_runs_out_reports_and_recovers(d, k):
    from decode_dsa_kv_gb300 import _abi
    B, H = 2, 128
    qb = wl.normal_bf16(B * H, 576, 91, 9, k, 0).reshape(B, H, 576)
    rows = wl.normal_bf16(B * k, 576, 92, 9, k, 0).reshape(B, k, 576)
    q = torch.from_numpy(qb.view(np.int16)).cuda()
    sel = torch.from_numpy(rows.view(np.int16)).cuda()
    scale = 1 / math.sqrt(576)
    d.ts_set_wait_limit_ns(1)
    try:
        _, bits = _sfa(d, q, sel, B, H, k, scale)
    finally:
        d.ts_set_wait_limit_ns(0)
    assert bits & _abi.TS_DEVERR_TIMEOUT, bits
    for _ in range(2):   # the context is usable and the default limit computes
        out, bits = _sfa(d, q, sel, B, H, k, scale)
        assert bits == 0
        got = out.cpu().view(torch.int16).numpy().view(np.uint16)
        for b in range(B):
            o, _ = oracle.sfa_decode(qb[b], rows[b], scale)
            a, rel = sfa_errors(got[b], oracle.round_to_bf16_bits(o))
            assert a <= SFA_ABS_TOL and rel <= SFA_MEAN_REL_TOL, (b, a, rel)


@pytest.mark.parametrize("layout", ["selection", "staged"])
def test_group_step_orders_streams_under_delays(d, layout):
    # small pools (256 sets x 16 ways) over 16,384-position contexts, so sets
    # evict from the second step on and code-2 installs (victim slots read as
    # hits in the same step) are common
    w = wl.scaled(wl.DECODE_BATCH, B=2, ctx=16384, S=256)
    T = 7
    staged = layout == "staged"
    lens = wl.ctx_lens(w)
    host = d.HostKV(w.layers, w.B, w.ctx_stride)
    wl.fill_host_kv(w, host.array)
    g = d.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host, layout=layout)
    stream = wl.ScoreStream(w)
    scores = np.stack([stream.next() for _ in range(T)])
    qs = np.stack([wl.queries(w, t) for t in range(T)])
    scores_d = torch.from_numpy(scores).cuda()
    q_d = torch.from_numpy(qs.view(np.int16)).cuda()
    # what each step's attention read: the selection buffers, or the staged rows
    rows = g.pool[:, :, w.P:] if staged else g.sel
    snap = {"ids": torch.empty((T, w.B, w.k), dtype=torch.int32, device="cuda"),
            "src": torch.empty((T, w.B, w.k), dtype=torch.int32, device="cuda"),
            "rows": torch.empty((T,) + tuple(rows.shape), dtype=torch.int16, device="cuda"),
            "out": torch.empty((T,) + tuple(g.out.shape), dtype=torch.bfloat16, device="cuda"),
            "install": torch.empty((T, w.B, w.k), dtype=torch.uint8, device="cuda"),
            "mc": torch.empty((T, w.B), dtype=torch.int32, device="cuda")}
    torch.cuda.synchronize()
    delayed = (g.side, g.gstream, g.main) + tuple(g.lstreams[1:2])
    for t in range(T):
        # about 2 ms of spinning ahead of this step's work on one stream:
        # the refill (then the next plan must wait for it), the gather (the
        # attention and the refill must wait), the top-k, plan and
        # attention (the gather must wait for the plan; with the staged layout
        # the refill must wait for the attention), or (streamed) layer 1's
        # attention stream (the later layers, that layer's refill and the
        # next step's plan must wait for it)
        with torch.cuda.stream(delayed[t % len(delayed)]):
            torch.cuda._sleep(4_000_000)
        g.step(scores_d[t], q_d[t])
        with torch.cuda.stream(g.main):   # after the step's last attention
            snap["ids"][t].copy_(g.ids)
            snap["src"][t].copy_(g.src_map)
            snap["rows"][t].copy_(rows)
            snap["out"][t].copy_(g.out)
            snap["install"][t].copy_(g.install)
            snap["mc"][t].copy_(g.miss_count)
    assert g.synchronize() == 0
    snap = {k: v.cpu() for k, v in snap.items()}
    scale = 1 / math.sqrt(576)
    ws_bytes = d.sfa_workspace_size(1, w.H, w.k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    deferred = 0
    for b in range(w.B):
        st = oracle.init_state(w.layers, w.S, w.W)
        for t in range(T):
            r = oracle.decode_step(st, scores[t, b], int(lens[b]), w.k, w.S, w.W,
                                   host.array[:, b], qs[t, :, b], scale, with_sfa=False)
            plan = r["plan"]
            M = plan.miss_count
            assert np.array_equal(snap["ids"][t, b].numpy(), r["ids"]), (t, b)
            assert np.array_equal(snap["src"][t, b].numpy(), plan.src_map), (t, b)
            assert int(snap["mc"][t, b]) == M
            assert np.array_equal(snap["install"][t, b, :M].numpy(), plan.install_code)
            deferred += int(np.sum(plan.install_code == 2))
            for l in range(w.layers):
                got_rows = snap["rows"][t, l, b].numpy().view(np.uint16)
                if staged:
                    assert np.array_equal(got_rows[plan.miss_pos], host.array[l, b][plan.miss_ids])
                else:
                    assert np.array_equal(got_rows, r["sel"][l]), (t, b, l)
            # the attention read exactly the oracle's rows: bit-exact against
            # the selection kernel over them, and within tolerance
            out = torch.empty((1, w.H, 512), dtype=torch.bfloat16, device="cuda")
            qb = torch.from_numpy(np.ascontiguousarray(qs[t, 3, b:b + 1]).view(np.int16)).cuda()
            selb = torch.from_numpy(np.ascontiguousarray(r["sel"][3][None]).view(np.int16)).cuda()
            assert d.sfa_mla_decode(qb, selb, 1, w.H, w.k, scale, out, None, ws, ws_bytes,
                                    err) == 0
            assert d.ts_read_error(err) == 0
            assert torch.equal(snap["out"][t, 3, b].view(torch.int16),
                               out[0].cpu().view(torch.int16)), (t, b)
            o, _ = oracle.sfa_decode(qs[t, 3, b], r["sel"][3], scale)
            got = snap["out"][t, 3, b].view(torch.int16).numpy().view(np.uint16)
            a, rel = sfa_errors(got, oracle.round_to_bf16_bits(o))
            assert a <= SFA_ABS_TOL and rel <= SFA_MEAN_REL_TOL, (t, b, a, rel)
        # the pool after the last step: metadata and every layer's rows
        assert np.array_equal(g.tags[b].cpu().numpy(), st.tags)
        assert np.array_equal(g.fifo_ptr[b].cpu().numpy(), st.fifo_ptr)
        for l in range(w.layers):
            assert np.array_equal(g.pool[l, b, :w.P].cpu().numpy().view(np.uint16), st.pool[l]), \
                (b, l)
    assert deferred > 0   # installs that had to wait for the layer's reads occurred
    host.close()


@pytest.mark.parametrize("layout,mixed", [("selection", False), ("staged", False),
                                          ("staged", True)])
def test_host_io_step_equals_device_input_step(d, layout, mixed):
    # dsa_group_step_host copies the inputs in and the output out inside the
    # step (the queries beside the top-k and plan, into a staging half chosen
    # by step parity; each layer's output on the side stream, which the next
    # step's attention of that layer waits for before it overwrites the
    # output): steps enqueued back to back without a sync give the same plan,
    # pool and attention output as steps on device-resident inputs. `mixed`:
    # host-I/O steps alternate with device-input steps on the same group.
    from decode_dsa_kv_gb300 import PinnedHost
    w = wl.scaled(wl.DECODE_BATCH, B=2, ctx=16384, S=256)
    T = 6
    lens = wl.ctx_lens(w)
    host = d.HostKV(w.layers, w.B, w.ctx_stride)
    wl.fill_host_kv(w, host.array)
    stream = wl.ScoreStream(w)
    scores = np.stack([stream.next() for _ in range(T)])
    qs = np.stack([wl.queries(w, t) for t in range(T)])
    s_pin = PinnedHost(scores.shape, np.float32)
    q_pin = PinnedHost(qs.shape, np.int16)
    o_pin = PinnedHost((T, w.layers, w.B, w.H, 512), np.int16)
    s_pin.array[...] = scores
    q_pin.array[...] = qs.view(np.int16)
    ga = d.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host, layout=layout)
    gb = d.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host, layout=layout)
    s_b, q_b, o_b = scores[0].nbytes, qs[0].nbytes, o_pin.array[0].nbytes
    outs = torch.empty((T,) + tuple(gb.out.shape), dtype=torch.bfloat16, device="cuda")
    scores_d = torch.from_numpy(scores).cuda()
    q_d = torch.from_numpy(qs.view(np.int16)).cuda()
    outs_a = torch.empty((T,) + tuple(ga.out.shape), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    for t in range(T):
        if mixed and t % 2:
            ga.step(scores_d[t], q_d[t])
            with torch.cuda.stream(ga.main):
                outs_a[t].copy_(ga.out)
        else:
            ga.step_host(s_pin.dev + t * s_b, q_pin.dev + t * q_b, o_pin.dev + t * o_b)
    torch.cuda.synchronize()
    for t in range(T):
        gb.step(scores_d[t], q_d[t])
        with torch.cuda.stream(gb.main):
            outs[t].copy_(gb.out)
    assert ga.synchronize() == 0 and gb.synchronize() == 0
    for t in range(T):
        got = (outs_a[t].cpu().view(torch.int16).numpy() if mixed and t % 2
               else o_pin.array[t]).view(np.uint16)
        want = outs[t].cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, want), t
    assert torch.equal(ga.tags, gb.tags) and torch.equal(ga.pool, gb.pool)
    assert torch.equal(ga.ids, gb.ids) and torch.equal(ga.src_map, gb.src_map)
    for pin in (s_pin, q_pin, o_pin):
        pin.close()
    host.close()


@pytest.mark.parametrize("w", [wl.scaled(wl.DECODE_BATCH, B=4, ctx=16384, S=256),
                               wl.scaled(wl.LARGE_BATCH, B=8, ctx=8192, S=128)])
def test_streamed_attention_wait_that_runs_out_reports_and_recovers(d, w):
    # streamed attention: with the wait limit at 1 ns every attention CTA
    # gives up waiting for its request's rows at once; the step reports
    # TS_DEVERR_TIMEOUT through the error word (no trap, no hang), the gather
    # and the refills still complete, and the steps after it, at the default
    # limit, equal those of a group that never timed out (outputs and pool,
    # bit for bit)
    from decode_dsa_kv_gb300 import _abi
    lens = wl.ctx_lens(w)
    host = d.HostKV(w.layers, w.B, w.ctx_stride)
    wl.fill_host_kv(w, host.array)
    ga = d.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host,
                       layout="staged")
    gb = d.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host,
                       layout="staged")
    assert ga.arrived is not None
    stream = wl.ScoreStream(w)
    for t in range(5):
        scores = torch.from_numpy(stream.next()).cuda()
        q = torch.from_numpy(wl.queries(w, t).view(np.int16)).cuda()
        if t == 2:
            d.ts_set_wait_limit_ns(1)
            try:
                ga.step(scores, q)
                bits = ga.synchronize()
            finally:
                d.ts_set_wait_limit_ns(0)
            assert bits & _abi.TS_DEVERR_TIMEOUT, bits
        else:
            ga.step(scores, q)
            assert ga.synchronize() == 0, t
        gb.step(scores, q)
        assert gb.synchronize() == 0, t
        assert torch.equal(ga.pool, gb.pool), t
        if t != 2:
            assert torch.equal(ga.out.view(torch.int16), gb.out.view(torch.int16)), t
    host.close()
