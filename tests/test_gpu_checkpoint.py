"""Checkpoint and resume of a group's pool state: a group that loads another
group's state() mid-run continues bit for bit as the original does, and the
oracle resumed from the same host arrays (one request's tags, pointers and
slot rows) plans each following step exactly as the device does."""
import math

import numpy as np
import pytest

import oracle
import workload as wl
from _util import ensure_library

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def d():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()
    import decode_dsa_kv_gb300 as d
    return d


@pytest.mark.parametrize("layout", ["selection", "staged"])
def test_resumed_group_and_oracle_continue_as_the_original(d, layout):
    w = wl.scaled(wl.DECODE_BATCH, B=2, ctx=16384, S=256)
    T, T0 = 6, 3
    lens = wl.ctx_lens(w)
    host = d.HostKV(w.layers, w.B, w.ctx_stride)
    wl.fill_host_kv(w, host.array)
    stream = wl.ScoreStream(w)
    scores = np.stack([stream.next() for _ in range(T)])
    qs = np.stack([wl.queries(w, t) for t in range(T)])
    scores_d = torch.from_numpy(scores).cuda()
    q_d = torch.from_numpy(qs.view(np.int16)).cuda()
    g1 = d.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host, layout=layout)
    for t in range(T0):
        g1.step(scores_d[t], q_d[t])
    st = g1.state()
    assert st["pool"].shape == (w.layers, w.B, w.P, 576)
    g2 = d.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host, layout=layout)
    g2.load_state(st)
    resumed = [oracle.RequestState(pool=st["pool"][:, b].view(np.uint16).copy(),
                                   tags=st["tags"][b].copy(),
                                   fifo_ptr=st["fifo_ptr"][b].copy())
               for b in range(w.B)]
    scale = 1 / math.sqrt(576)
    for t in range(T0, T):
        g1.step(scores_d[t], q_d[t])
        g2.step(scores_d[t], q_d[t])
        assert g1.synchronize() == 0 and g2.synchronize() == 0
        assert torch.equal(g1.out.view(torch.int16), g2.out.view(torch.int16)), t
        assert torch.equal(g1.tags, g2.tags) and torch.equal(g1.fifo_ptr, g2.fifo_ptr), t
        assert torch.equal(g1.pool[:, :, :w.P], g2.pool[:, :, :w.P]), t
        for b in range(w.B):
            r = oracle.decode_step(resumed[b], scores[t, b], int(lens[b]), w.k, w.S, w.W,
                                   host.array[:, b], qs[t, :, b], scale, with_sfa=False)
            assert np.array_equal(g2.src_map[b].cpu().numpy(), r["plan"].src_map), (t, b)
            assert np.array_equal(g2.tags[b].cpu().numpy(), resumed[b].tags), (t, b)
            assert np.array_equal(g2.pool[:, b, :w.P].cpu().numpy().view(np.uint16),
                                  resumed[b].pool), (t, b)
    host.close()


def test_load_state_refuses_another_shape(d):
    w = wl.scaled(wl.TINY, B=1)
    lens = wl.ctx_lens(w)
    host = d.HostKV(w.layers, w.B, w.ctx_stride)
    g = d.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host)
    st = g.state()
    st["tags"] = np.zeros((w.B, w.P + 1), np.int32)
    with pytest.raises(ValueError):
        g.load_state(st)
    host.close()
